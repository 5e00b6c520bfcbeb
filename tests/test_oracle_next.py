"""Pins of the oracle's next rows against facts fixed outside the oracle itself.

Cross-attention keys/values ("whisper 0.9.0 API", model.nu, wh_prepare_cross):
- A permutation matrix moves columns (a transposed weight would move them the other way).
- A zero memory gives K = 0 and V = bv (the bias belongs to V, not to K).
- A zero V projection gives V = bv in every row.
- A projection built from a known rank-1 pair gives K = (mem a) b^T.

Shorter encoder context (the "whisper" package page, "Serving": whisper.cpp's audio_ctx):
- n_ctx = 1500 is the full encoder.
- Frames past 2 n_ctx are never read.
- The span's end is zero-padded like the end of a window. So the stem equals the full stem
  of a log-mel whose frames past 2 n_ctx are zero, and rows before the last agree with the
  full-window stem.
"""
import numpy as np
import pytest

from oracle import whisper_ref as R
from whisper_audio_encoder_gb300 import synth
from whisper_audio_encoder_gb300.configs import CONFIGS

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.fixture(scope="module")
def mem():
    rng = np.random.default_rng(3)
    return rng.standard_normal((50, 16))


def test_cross_kv_moves_columns_by_the_permutation(mem):
    d = mem.shape[1]
    perm = np.roll(np.arange(d), 3)                  # not an involution: W and W^T differ
    w = np.zeros((d, d))
    w[np.arange(d), perm] = 1.0                      # out column o reads input column perm[o]
    k, v = R.cross_kv(mem, w, w)
    np.testing.assert_array_equal(k, mem[:, perm])
    np.testing.assert_array_equal(v, mem[:, perm])
    assert not np.allclose(k, mem @ w)               # the transposed operand gives another answer


def test_cross_kv_bias_is_on_v_only(mem):
    d = mem.shape[1]
    rng = np.random.default_rng(4)
    wk, wv, bv = rng.standard_normal((d, d)), rng.standard_normal((d, d)), rng.standard_normal(d)
    k, v = R.cross_kv(np.zeros_like(mem), wk, wv, bv)
    assert np.all(k == 0.0)
    np.testing.assert_array_equal(v, np.broadcast_to(bv, v.shape))
    k2, v2 = R.cross_kv(mem, wk, np.zeros((d, d)), bv)
    np.testing.assert_array_equal(v2, np.broadcast_to(bv, v2.shape))
    k3, _ = R.cross_kv(mem, wk, wv, None)
    np.testing.assert_array_equal(k2, k3)


def test_cross_kv_rank_one_projection(mem):
    d = mem.shape[1]
    rng = np.random.default_rng(5)
    a, b = rng.standard_normal(d), rng.standard_normal(d)
    w = np.outer(b, a)                               # y[o] = b[o] * (a . x)
    k, _ = R.cross_kv(mem, w, w)
    np.testing.assert_allclose(k, np.outer(mem @ a, b), rtol=1e-12, atol=1e-12)


@pytest.fixture(scope="module")
def tiny():
    cfg = CONFIGS[0]
    w = synth.weights(cfg)
    pcm = synth.waveform(cfg, 0)
    mel = R.log_mel(pcm, cfg.n_mels)
    return cfg, w, mel


def test_encoder_ctx_full_context_is_the_encoder(tiny):
    cfg, w, mel = tiny
    np.testing.assert_array_equal(R.encoder_ctx(mel, w, cfg.n_head, 1500), R.encoder(mel, w, cfg.n_head))


@pytest.mark.parametrize("n_ctx", [500, 37])
def test_encoder_ctx_reads_only_its_span(tiny, n_ctx):
    cfg, w, mel = tiny
    out = R.encoder_ctx(mel, w, cfg.n_head, n_ctx)
    assert out.shape == (n_ctx, cfg.d_model)
    other = mel.copy()
    other[2 * n_ctx:] = np.random.default_rng(9).standard_normal(other[2 * n_ctx:].shape)
    np.testing.assert_array_equal(R.encoder_ctx(other, w, cfg.n_head, n_ctx), out)


@pytest.mark.parametrize("n_ctx", [500, 37])
def test_encoder_ctx_zero_pads_the_end_of_its_span(tiny, n_ctx):
    cfg, w, mel = tiny
    short = R.encoder_stem(mel[: 2 * n_ctx], w)
    zeroed = mel.copy()
    zeroed[2 * n_ctx:] = 0.0
    full_zeroed = R.encoder_stem(zeroed, w)[:n_ctx]
    np.testing.assert_allclose(short, full_zeroed, rtol=1e-12, atol=1e-12)
    full = R.encoder_stem(mel, w)[:n_ctx]
    np.testing.assert_allclose(short[:-1], full[:-1], rtol=1e-12, atol=1e-12)  # receptive field inside the span
    assert np.max(np.abs(short[-1] - full[-1])) > 1e-6     # the last position sees the padding


# ---- one-query attention of a decoder step ------------------------------------------------
def test_attend_one_equal_keys_give_the_mean_of_v():
    rng = np.random.default_rng(20)
    n_head, n = 3, 17
    q = rng.standard_normal(64 * n_head)
    k = np.tile(rng.standard_normal(64 * n_head), (n, 1))
    v = rng.standard_normal((n, 64 * n_head))
    np.testing.assert_allclose(R.attend_one(q, k, v, n_head), v.mean(axis=0), rtol=1e-12, atol=1e-12)


def test_attend_one_dominant_key_selects_its_value():
    rng = np.random.default_rng(21)
    n_head, n, j = 2, 40, 23
    k = rng.standard_normal((n, 64 * n_head)) * 0.01
    q = np.zeros(64 * n_head)
    q[0], q[64] = 1.0, 1.0
    k[j, 0], k[j, 64] = 800.0, 800.0        # score 100 above the rest after the 1/8 scale
    v = rng.standard_normal((n, 64 * n_head))
    np.testing.assert_allclose(R.attend_one(q, k, v, n_head), v[j], rtol=1e-12, atol=1e-12)


def test_attend_one_ignores_key_order_single_key_and_empty():
    rng = np.random.default_rng(22)
    n_head, n = 4, 33
    q, k, v = rng.standard_normal(256), rng.standard_normal((n, 256)), rng.standard_normal((n, 256))
    perm = rng.permutation(n)
    np.testing.assert_allclose(R.attend_one(q, k[perm], v[perm], n_head), R.attend_one(q, k, v, n_head),
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(R.attend_one(q, k[:1], v[:1], n_head), v[0], rtol=1e-12, atol=1e-12)
    assert np.all(R.attend_one(q, k[:0], v[:0], n_head) == 0.0)


def test_attend_one_matches_torch_sdpa():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(23)
    n_head, n = 5, 300
    q, k, v = rng.standard_normal(320), rng.standard_normal((n, 320)), rng.standard_normal((n, 320))
    qt = torch.from_numpy(q).reshape(1, n_head, 1, 64)
    kt = torch.from_numpy(k).reshape(n, n_head, 64).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).reshape(n, n_head, 64).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).reshape(-1).numpy()
    np.testing.assert_allclose(R.attend_one(q, k, v, n_head), ref, rtol=1e-10, atol=1e-12)


# ---- upstream front end: long clips and resampling ------------------------------------------
def test_long_clip_windows_cover_the_clip_and_pad_the_last():
    x = np.arange(2 * 480000 + 1234, dtype=np.float32)
    w = R.long_clip_windows(x)
    assert len(w) == 3 and all(v.shape == (480000,) for v in w)
    np.testing.assert_array_equal(np.concatenate(w)[: x.shape[0]], x)
    assert np.all(w[2][1234:] == 0.0)
    assert R.long_clip_windows(np.zeros(0, np.float32)) == []


@pytest.mark.parametrize("rate", [44100, 48000, 22050, 8000, 11025, 32000, 24000])
def test_resample_matches_scipy_resample_poly(rate):
    signal = pytest.importorskip("scipy.signal")
    from math import gcd
    rng = np.random.default_rng(rate)
    x = rng.standard_normal(rate // 4 + 37)
    g = gcd(16000, rate)
    ref = signal.resample_poly(x, 16000 // g, rate // g)
    got = R.resample_to_16k(x, rate)
    assert got.shape == ref.shape
    np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-10)


def test_resample_at_16k_is_the_identity():
    x = np.random.default_rng(1).standard_normal(5000)
    np.testing.assert_allclose(R.resample_to_16k(x, 16000), x, rtol=0, atol=1e-12)


@pytest.mark.parametrize("rate", [44100, 8000])
def test_resample_keeps_a_passband_tone(rate):
    """A 1 kHz tone sampled at `rate` comes out as the same tone at 16 kHz (away from the
    clip's ends, within the Kaiser-window filter's passband ripple)."""
    n = rate // 2
    x = np.cos(2 * np.pi * 1000.0 * np.arange(n) / rate)
    y = R.resample_to_16k(x, rate)
    j = np.arange(y.shape[0])
    ref = np.cos(2 * np.pi * 1000.0 * j / 16000.0)
    mid = slice(400, y.shape[0] - 400)
    assert np.max(np.abs(y[mid] - ref[mid])) < 5e-3
