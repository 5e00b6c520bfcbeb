"""Seeded synthetic inputs shared by the tests, the benchmark and the CPU oracle runs.

This module holds input generation only -- waveforms and random weights -- and none of the
encoder's arithmetic.  Every array is drawn from numpy's PCG64 with a fixed seed:
  waveform of window w in workload c : seed (1000 * c + w)
  weight tensor t of layer l         : seed sequence (7 + c, l, t)
so any single window or any single layer can be regenerated on its own.

Matrices are rounded to bfloat16 (round to nearest even) here, once, so that the GPU path
and the oracle see exactly the same weight values.
"""
import numpy as np

from .configs import N_SAMPLES, N_CTX, N_TEXT_CTX, SAMPLE_RATE, EncoderConfig


# ----------------------------------------------------------------------------------------
# bfloat16 helpers (storage format conversion only)
# ----------------------------------------------------------------------------------------
def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + r) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Values of `a` rounded to the nearest bfloat16, returned as float32."""
    return bf16_to_f32(bf16_bits(a))


# ----------------------------------------------------------------------------------------
# waveforms
# ----------------------------------------------------------------------------------------
def _sines(rng: np.random.Generator, n: int) -> np.ndarray:
    t = np.arange(n, dtype=np.float64) / SAMPLE_RATE
    f = rng.uniform(100.0, 4000.0, size=5)
    ph = rng.uniform(0.0, 2.0 * np.pi, size=5)
    x = np.zeros(n, dtype=np.float64)
    for fi, pi in zip(f, ph):
        x += 0.1 * np.sin(2.0 * np.pi * fi * t + pi)
    x += rng.normal(0.0, 0.01, size=n)
    return x.astype(np.float32)


def _pink_noise(rng: np.random.Generator, n: int) -> np.ndarray:
    white = rng.standard_normal(n)
    spec = np.fft.rfft(white)
    k = np.arange(spec.shape[0], dtype=np.float64)
    k[0] = np.inf                       # no DC
    spec = spec / np.sqrt(k)
    pink = np.fft.irfft(spec, n=n)
    return pink / np.sqrt(np.mean(pink ** 2))


def _speech_like(rng: np.random.Generator, n: int) -> np.ndarray:
    """A harmonic stack on a slowly vibrating pitch, syllable-rate amplitude modulation and
    pink noise 20 dB down, scaled to RMS 0.05."""
    t = np.arange(n, dtype=np.float64) / SAMPLE_RATE
    f0 = rng.uniform(80.0, 250.0)
    rate = rng.uniform(3.0, 6.0)
    ph0 = rng.uniform(0.0, 2.0 * np.pi)
    # phase of f0 * (1 + 0.03 sin(2 pi 5 t)), integrated in closed form
    phase = 2.0 * np.pi * f0 * (t - 0.03 / (2.0 * np.pi * 5.0) * np.cos(2.0 * np.pi * 5.0 * t)) + ph0
    x = np.zeros(n, dtype=np.float64)
    k = 1
    while k * f0 <= 4000.0:
        x += np.sin(k * phase + rng.uniform(0.0, 2.0 * np.pi)) / k
        k += 1
    env = (0.5 + 0.5 * np.sin(2.0 * np.pi * rate * t + rng.uniform(0.0, 2.0 * np.pi))) ** 2
    x *= env
    x /= np.sqrt(np.mean(x ** 2))
    x += 0.1 * _pink_noise(rng, n)      # -20 dB relative
    x *= 0.05 / np.sqrt(np.mean(x ** 2))
    return x.astype(np.float32)


def waveform(cfg: EncoderConfig, window: int, n: int = N_SAMPLES) -> np.ndarray:
    """One synthetic 16 kHz clip (float32 [n]) for window `window` of workload `cfg`."""
    rng = np.random.Generator(np.random.PCG64(1000 * cfg.index + window))
    x = _sines(rng, n) if cfg.waveform == "sines" else _speech_like(rng, n)
    if window in cfg.silent_windows:
        x[144_000:] = 0.0               # a 9-s clip zero-padded to 30 s
    return x


def waveforms(cfg: EncoderConfig, windows=None) -> np.ndarray:
    windows = range(cfg.batch) if windows is None else windows
    return np.stack([waveform(cfg, w) for w in windows])


# ----------------------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------------------
_TENSORS = ["wq", "bq", "wk", "wv", "bv", "wo", "bo", "w1", "b1", "w2", "b2",
            "ln1_g", "ln1_b", "ln2_g", "ln2_b"]


def _rng(cfg: EncoderConfig, layer: int, tensor: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([7 + cfg.index, layer, tensor]))


def _normal(rng, shape, std):
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def _gamma(cfg, rng, d):
    if cfg.ln_gamma_jitter:
        return (1.0 + rng.uniform(-cfg.ln_gamma_jitter, cfg.ln_gamma_jitter, size=d)).astype(np.float32)
    return np.ones(d, dtype=np.float32)


def layer_weights(cfg: EncoderConfig, layer: int) -> dict:
    """Weights of encoder block `layer`: matrices [out][in] (bf16 values as float32), vectors float32.
    There is no k bias: Whisper's k projection has none."""
    d, f = cfg.d_model, cfg.d_ff
    g = lambda name: _rng(cfg, 100 + layer, _TENSORS.index(name))
    return {
        "wq": bf16_round(_normal(g("wq"), (d, d), 0.02)), "bq": _normal(g("bq"), (d,), 0.01),
        "wk": bf16_round(_normal(g("wk"), (d, d), 0.02)),
        "wv": bf16_round(_normal(g("wv"), (d, d), 0.02)), "bv": _normal(g("bv"), (d,), 0.01),
        "wo": bf16_round(_normal(g("wo"), (d, d), 0.02)), "bo": _normal(g("bo"), (d,), 0.01),
        "w1": bf16_round(_normal(g("w1"), (f, d), 0.02)), "b1": _normal(g("b1"), (f,), 0.01),
        "w2": bf16_round(_normal(g("w2"), (d, f), 0.02)), "b2": _normal(g("b2"), (d,), 0.01),
        "ln1_g": _gamma(cfg, g("ln1_g"), d), "ln1_b": np.zeros(d, np.float32),
        "ln2_g": _gamma(cfg, g("ln2_g"), d), "ln2_b": np.zeros(d, np.float32),
    }


def stem_weights(cfg: EncoderConfig) -> dict:
    """Conv stem (PyTorch Conv1d layout [c_out][c_in][3]), stored positions and final norm."""
    d, M = cfg.d_model, cfg.n_mels
    return {
        "conv1_w": bf16_round(_normal(_rng(cfg, 0, 0), (d, M, 3), 0.02)),
        "conv1_b": _normal(_rng(cfg, 0, 1), (d,), 0.01),
        "conv2_w": bf16_round(_normal(_rng(cfg, 0, 2), (d, d, 3), 0.02)),
        "conv2_b": _normal(_rng(cfg, 0, 3), (d,), 0.01),
        "pos": _normal(_rng(cfg, 0, 4), (N_CTX, d), 0.02),
        "lnf_g": _gamma(cfg, _rng(cfg, 0, 5), d),
        "lnf_b": np.zeros(d, np.float32),
    }


def weights(cfg: EncoderConfig, layers=None) -> dict:
    """All weights: the stem dict plus "layers": a list of per-block dicts."""
    w = stem_weights(cfg)
    layers = range(cfg.n_layer) if layers is None else layers
    w["layers"] = [layer_weights(cfg, l) for l in layers]
    return w


def cross_weights(cfg: EncoderConfig, n_layer=None) -> list:
    """Cross-attention k/v projections of the decoder layers (Whisper's decoder has as many
    layers as its encoder): wk, wv N(0, 0.02) rounded to bf16, bv N(0, 0.01).  Layer l's
    tensors use the seed sequence (7 + c, 1000 + l, t)."""
    n = cfg.n_layer if n_layer is None else n_layer
    d = cfg.d_model
    out = []
    for l in range(n):
        out.append({"wk": bf16_round(_normal(_rng(cfg, 1000 + l, 0), (d, d), 0.02)),
                    "wv": bf16_round(_normal(_rng(cfg, 1000 + l, 1), (d, d), 0.02)),
                    "bv": _normal(_rng(cfg, 1000 + l, 2), (d,), 0.01).astype(np.float32)})
    return out


def random_weights(n_mels, d_model, n_layer, d_ff, seed, ln_random=False) -> dict:
    """Weights of an arbitrary (test-sized) encoder, same distributions as the workloads.
    With ln_random the LayerNorm gamma/beta are drawn too (so a swapped or dropped
    parameter shows up in a comparison)."""
    cfg = EncoderConfig("custom", n_mels, d_model, max(1, d_model // 64), n_layer, d_ff, 1,
                        "sines", index=seed)
    w = weights(cfg)
    if ln_random:
        rng = np.random.Generator(np.random.PCG64([seed, 999]))
        for lw in w["layers"]:
            for k in ("ln1_g", "ln2_g"):
                lw[k] = (1.0 + 0.2 * rng.standard_normal(d_model)).astype(np.float32)
            for k in ("ln1_b", "ln2_b"):
                lw[k] = (0.1 * rng.standard_normal(d_model)).astype(np.float32)
        w["lnf_g"] = (1.0 + 0.2 * rng.standard_normal(d_model)).astype(np.float32)
        w["lnf_b"] = (0.1 * rng.standard_normal(d_model)).astype(np.float32)
    return w


# ----------------------------------------------------------------------------------------
# decoder (one decode step): weights, cross-attention keys/values, self-attention caches
# ----------------------------------------------------------------------------------------
_DEC_TENSORS = ["ln1_g", "ln1_b", "wq", "bq", "wk", "wv", "bv", "wo", "bo", "lnx_g", "lnx_b", "xwq", "xbq",
                "xwo", "xbo", "ln2_g", "ln2_b", "w1", "b1", "w2", "b2"]


def decoder_layer_weights(cfg: EncoderConfig, layer: int, ln_random: bool = False) -> dict:
    """Decoder block `layer` (seed sequence (7 + c, 2000 + layer, t)): self-attention q/k/v/out
    (no k bias), the cross-attention query and output projections (its k/v projections are
    cross_weights), fc1/fc2, and three LayerNorms (ln1, lnx before the cross-attention,
    ln2).  Matrices N(0, 0.02) rounded to bf16, biases N(0, 0.01); LayerNorm gamma as the
    encoder's, beta 0 -- or, with ln_random, gamma 1 + N(0, 0.2) and beta N(0, 0.1) so that a
    swapped or dropped norm parameter shows in a comparison."""
    d, f = cfg.d_model, cfg.d_ff
    g = lambda name: _rng(cfg, 2000 + layer, _DEC_TENSORS.index(name))
    w = {}
    for name in ("wq", "wk", "wv", "wo", "xwq", "xwo"):
        w[name] = bf16_round(_normal(g(name), (d, d), 0.02))
    w["w1"] = bf16_round(_normal(g("w1"), (f, d), 0.02))
    w["w2"] = bf16_round(_normal(g("w2"), (d, f), 0.02))
    for name in ("bq", "bv", "bo", "xbq", "xbo", "b2"):
        w[name] = _normal(g(name), (d,), 0.01)
    w["b1"] = _normal(g("b1"), (f,), 0.01)
    for ln in ("ln1", "lnx", "ln2"):
        if ln_random:
            w[ln + "_g"] = (1.0 + _normal(g(ln + "_g"), (d,), 0.2)).astype(np.float32)
            w[ln + "_b"] = _normal(g(ln + "_b"), (d,), 0.1)
        else:
            w[ln + "_g"] = _gamma(cfg, g(ln + "_g"), d)
            w[ln + "_b"] = np.zeros(d, np.float32)
    return w


def decoder_weights(cfg: EncoderConfig, n_layer=None, n_vocab=None, n_text_ctx: int = N_TEXT_CTX,
                    ln_random: bool = False) -> dict:
    """All decoder weights of a decode step: "tok_embd" [n_vocab][d] (bf16 values; also the
    output projection, Whisper ties them), "dec_pos" [n_text_ctx][d] float32, "layers" and
    the final norm "lnf_g" / "lnf_b"."""
    d = cfg.d_model
    n_layer = cfg.n_layer if n_layer is None else n_layer
    n_vocab = cfg.n_vocab if n_vocab is None else n_vocab
    w = {"tok_embd": bf16_round(_normal(_rng(cfg, 1999, 0), (n_vocab, d), 0.02)),
         "dec_pos": _normal(_rng(cfg, 1999, 1), (n_text_ctx, d), 0.02),
         "layers": [decoder_layer_weights(cfg, l, ln_random) for l in range(n_layer)]}
    if ln_random:
        w["lnf_g"] = (1.0 + _normal(_rng(cfg, 1999, 2), (d,), 0.2)).astype(np.float32)
        w["lnf_b"] = _normal(_rng(cfg, 1999, 3), (d,), 0.1)
    else:
        w["lnf_g"] = _gamma(cfg, _rng(cfg, 1999, 2), d)
        w["lnf_b"] = np.zeros(d, np.float32)
    return w


def cross_kv_values(cfg: EncoderConfig, batch: int, n_ctx: int, n_layer=None, seed: int = 0) -> np.ndarray:
    """Stand-in cross-attention keys and values for a decode step, in wh_prepare_cross's
    layout: float32 (bf16 values) [n_layer][batch * n_ctx][2 d], K in columns 0..d-1 and V in
    d..2d-1.  N(0, 0.5): about the spread of K = mem Wk^T for a unit-variance memory and
    N(0, 0.02) weights at d = 384..1280."""
    n_layer = cfg.n_layer if n_layer is None else n_layer
    rng = np.random.Generator(np.random.PCG64([7 + cfg.index, 3000, seed]))
    return bf16_round(_normal(rng, (n_layer, batch * n_ctx, 2 * cfg.d_model), 0.5))
