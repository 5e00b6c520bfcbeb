"""End-to-end parity: GPU front end + encoder (wh_frontend + wh_encode through the C ABI)
against the oracle on the five workloads at their full batch sizes, compared window by
window on sampled windows (the oracle runs one window at a time in float64).

Bar: log-mel max-abs <= 1e-3; encoder output max-abs <= 3e-2 and every frame's cosine
similarity >= 0.999."""
import numpy as np
import pytest
import torch

from oracle import whisper_ref as R
from whisper_audio_encoder_gb300 import build, configs, synth, wh

from helpers import ENC_ATOL, LOGMEL_ATOL, check_encoder, maxabs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build.build()
    wh.lib()



@pytest.mark.parametrize("idx,windows", [(0, [0]), (1, [0, 2, 7]), (2, [0, 15]), (3, [0, 31]), (4, [0, 15])])
def test_encoder_parity_on_workloads(idx, windows):
    cfg = configs.CONFIGS[idx]
    w = synth.weights(cfg)
    enc = wh.Encoder(cfg, w)
    pcm = synth.waveforms(cfg)
    mel_d = wh.wh_frontend(torch.from_numpy(pcm).cuda(), cfg.n_mels)
    out = enc.wh_encode(mel_d)
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    out = out.cpu().numpy()
    mel = mel_d.cpu().numpy()
    assert out.shape == (cfg.batch, 1500, cfg.d_model)
    assert np.isfinite(out).all()
    for win in windows:
        mel_ref, out_ref = R.encode_window(pcm[win], w, cfg.n_mels, cfg.n_head)
        assert maxabs(mel[win], mel_ref) <= LOGMEL_ATOL
        check_encoder(out[win], out_ref, f"{cfg.name} window {win}")


def test_encoder_with_random_layernorm_and_ragged_width():
    """A non-Whisper width (d = 128, 2 heads, 128 mels) with random LayerNorm gamma/beta, so
    a dropped or swapped LayerNorm parameter or a 128-wide tile path shows up."""
    cfg = configs.EncoderConfig("test-d128", 128, 128, 2, 2, 512, 3, "speech", index=2)
    w = synth.random_weights(128, 128, 2, 512, seed=21, ln_random=True)
    enc = wh.Encoder(cfg, w)
    pcm = synth.waveforms(cfg)
    out = enc.forward(torch.from_numpy(pcm).cuda()).cpu().numpy()
    for win in range(3):
        _, ref = R.encode_window(pcm[win], w, 128, 2)
        check_encoder(out[win], ref, f"window {win}")


def test_stem_only_encoder():
    """n_layer = 0: conv stem + positions + final LayerNorm."""
    cfg = configs.EncoderConfig("stem-only", 80, 384, 6, 0, 1536, 2, "sines", index=1)
    w = synth.random_weights(80, 384, 0, 1536, seed=4, ln_random=True)
    enc = wh.Encoder(cfg, w)
    mel = np.random.default_rng(2).uniform(-1, 1, (2, 3000, 80)).astype(np.float32)
    out = enc.wh_encode(torch.from_numpy(mel).cuda()).cpu().numpy()
    for b in range(2):
        check_encoder(out[b], R.encoder(mel[b].astype(np.float64), w, 6), f"stem window {b}")


def test_windows_are_independent():
    """The same window at two batch positions gives bit-identical memories, and changing one
    window does not change another (no cross-window leakage in any kernel)."""
    cfg = configs.CONFIGS[1]
    enc = wh.Encoder(cfg, synth.weights(cfg))
    pcm = synth.waveforms(cfg, windows=[3, 4, 3, 5])
    out1 = enc.forward(torch.from_numpy(pcm).cuda()).cpu().numpy()
    assert np.array_equal(out1[0], out1[2])
    pcm[1] *= 0.5
    out2 = enc.forward(torch.from_numpy(pcm).cuda()).cpu().numpy()
    assert np.array_equal(out1[0], out2[0]) and np.array_equal(out1[3], out2[3])
    assert not np.array_equal(out1[1], out2[1])


def test_encode_is_deterministic():
    cfg = configs.CONFIGS[0]
    enc = wh.Encoder(cfg, synth.weights(cfg))
    mel = wh.wh_frontend(torch.from_numpy(synth.waveforms(cfg)).cuda(), 80)
    a = enc.wh_encode(mel).cpu().numpy()
    b = enc.wh_encode(mel).cpu().numpy()
    assert np.array_equal(a, b)


def test_stream_k_fc2_is_deterministic_and_matches_whole_tiles():
    """fc2 of a large-v3-width block over 16 windows (470 tiles of 80 k-blocks on the resident
    CTA pairs) runs its last rounds stream-K: the k-blocks are shared evenly between the pairs
    and a tile cut between two pairs is summed in two pieces.  Two runs give the same bits; each
    window agrees with the same window encoded alone (whole tiles only: 30 tiles, one round)
    up to the rounding of the split sums and its bf16 re-roundings downstream; window 9
    matches the oracle."""
    cfg = configs.EncoderConfig("sk-1280", 128, 1280, 20, 2, 5120, 16, "speech", index=3)
    w = synth.random_weights(128, 1280, 2, 5120, seed=77, ln_random=True)
    enc = wh.Encoder(cfg, w)
    pcm = synth.waveforms(cfg)
    mel = wh.wh_frontend(torch.from_numpy(pcm).cuda(), 128)
    a = enc.wh_encode(mel).clone()
    b = enc.wh_encode(mel)
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    assert torch.equal(a, b)
    worst = 0.0
    for win in (0, 9, 15):
        one = enc.wh_encode(mel[win:win + 1].contiguous())
        torch.cuda.synchronize()
        worst = max(worst, (a[win] - one[0]).abs().max().item())
    # Both are valid evaluation orders of the same bf16-operand arithmetic, so they may differ
    # by what each may differ from the oracle (one flipped bf16 rounding of an activation
    # spreads through the next block); a dropped or doubled piece would be off by O(1).
    assert worst <= ENC_ATOL, f"stream-K vs whole tiles: max |diff| {worst:.3e}"
    _, ref = R.encode_window(pcm[9], w, 128, 20)
    check_encoder(a[9].cpu().numpy(), ref, "window 9")


@pytest.mark.parametrize("batch,windows", [(4, [0, 3]), (11, [0, 5, 10])])
def test_stream_k_shares_without_and_with_round_robin_rounds(batch, windows):
    """fc2 at large-v3 width, one block: 4 windows are 120 tiles (fewer than two rounds, so every
    k-block is shared out stream-K); 11 windows are 325 tiles (three round-robin rounds, then
    the last round and the remainder shared out).  Sampled windows against the oracle, and two
    runs bitwise equal."""
    cfg = configs.EncoderConfig(f"sk-b{batch}", 128, 1280, 20, 1, 5120, batch, "speech", index=3)
    w = synth.random_weights(128, 1280, 1, 5120, seed=80 + batch, ln_random=True)
    enc = wh.Encoder(cfg, w)
    pcm = synth.waveforms(cfg)
    mel = wh.wh_frontend(torch.from_numpy(pcm).cuda(), 128)
    a = enc.wh_encode(mel).clone()
    b = enc.wh_encode(mel)
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    assert torch.equal(a, b)
    out = a.cpu().numpy()
    for win in windows:
        _, ref = R.encode_window(pcm[win], w, 128, 20)
        check_encoder(out[win], ref, f"batch {batch}, window {win}")
