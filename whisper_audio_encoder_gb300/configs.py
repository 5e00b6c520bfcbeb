"""The five encoder workloads: model shapes, batch size and the kind of synthetic audio.

Shapes follow the Whisper family table of "How Audio Becomes Words: Whisper's Kernels
Step By Step On A CPU" (section "Tiny, Base, Small, Large: What Actually Changes"):
tiny 4 layers / 384 / 6 heads, base 6 / 512 / 8, small 12 / 768 / 12, large 32 / 1280 / 20
with 128 mel bins for large-v3.  The feed-forward width is 4 * d_model (the same page,
section "The Full Stitched Circuit", where the MLP widens d to four times d).  The first
workload is a one-block tiny-width encoder, the smallest case that still runs every kernel
of the path.
"""
from dataclasses import dataclass, field

N_SAMPLES = 480_000      # 30 s at 16 kHz
N_FRAMES = 3000          # STFT frames per window (hop 160)
N_CTX = 1500             # encoder positions after the stride-2 conv
SAMPLE_RATE = 16_000
N_TEXT_CTX = 448         # decoder positions (the self-attention cache capacity)


@dataclass(frozen=True)
class EncoderConfig:
    name: str
    n_mels: int
    d_model: int
    n_head: int
    n_layer: int
    d_ff: int
    batch: int
    waveform: str                      # "sines" or "speech"
    silent_windows: tuple = ()         # windows whose samples from 144000 on are exact zeros
    ln_gamma_jitter: float = 0.0       # LayerNorm gamma = 1 + U(-j, j)
    index: int = 0

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_head

    @property
    def n_vocab(self) -> int:
        """Decoder vocabulary: the multilingual tokenizer's 51865 ids; large-v3 has one more
        (an extra language token).  The pages read it from the checkpoint's header."""
        return 51866 if self.n_mels == 128 else 51865

    def flops_per_window(self) -> dict:
        """Algorithmic flops of one window, counted from the definition of each step
        (2 flops per multiply-add; attention counts q.k and p.v)."""
        T, F, d, M, L, f = N_CTX, N_FRAMES, self.d_model, self.n_mels, self.n_layer, self.d_ff
        conv1 = 2.0 * F * d * 3 * M
        conv2 = 2.0 * T * d * 3 * d
        gemm = L * (2.0 * T * d * 3 * d + 2.0 * T * d * d + 2.0 * T * d * f * 2)
        attn = L * 4.0 * T * T * d
        return {"conv1": conv1, "conv2": conv2, "gemm": gemm, "attn": attn,
                "total": conv1 + conv2 + gemm + attn}


CONFIGS = [
    EncoderConfig("tiny-width-1block", 80, 384, 6, 1, 1536, 1, "sines", index=0),
    EncoderConfig("whisper-tiny", 80, 384, 6, 4, 1536, 8, "sines", silent_windows=(0, 1), index=1),
    EncoderConfig("whisper-base", 80, 512, 8, 6, 2048, 16, "speech", index=2),
    EncoderConfig("whisper-small", 80, 768, 12, 12, 3072, 32, "speech", index=3),
    EncoderConfig("whisper-large-v3", 128, 1280, 20, 32, 5120, 16, "speech",
                  ln_gamma_jitter=0.05, index=4),
]

BY_NAME = {c.name: c for c in CONFIGS}
