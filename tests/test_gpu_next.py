"""GPU parity of the next rows, called through the C ABI, against the oracle.

wh_prepare_cross: the cross-attention keys/values of every decoder layer.
- Against the oracle fed the bf16-rounded memory: the bf16 GEMM bound, 2^-8 |ref| + 1e-3.
- Against the oracle fed the float32 memory: that bound plus the operand rounding,
  2^-9 sum_i |mem_i| |w_i|.
- Shapes: tiny and large widths, ragged row counts, and a full large-v3 decoder (32 layers,
  16 windows) on sampled rows.

wh_encode_ctx: the encoder over the first 2 n_ctx log-mel frames.
- n_ctx = 1500 is bitwise wh_encode.
- Shorter contexts are held to the encoder bar against the oracle's encoder_ctx.

wh_decode_attention: one query per (sequence, head), keys split across blocks and merged.
- Against the oracle's attend_one: bf16 output rounding, 2^-8 |ref| + 1e-4 max|v|.
- Layouts: dense caches, wh_prepare_cross's [K | V] rows, and a ragged self-attention cache
  with an empty sequence.
- Many splits: 20 000 keys.
"""
import numpy as np
import pytest
import torch

from oracle import whisper_ref as R
from whisper_audio_encoder_gb300 import build, configs, synth, wh

from helpers import bf16_round_np, check_encoder

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build.build()
    wh.lib()


def _check_cross(kv, mem, layers, rows, what):
    """kv: numpy float32 [n_layer][R][2d] from the GPU; mem float32 [R][d]; rows: indices."""
    d = mem.shape[1]
    m16 = bf16_round_np(mem).astype(np.float64)
    for l, lw in enumerate(layers):
        k_ref, v_ref = R.cross_kv(m16[rows], lw["wk"], lw["wv"], lw["bv"])
        got_k, got_v = kv[l][rows, :d], kv[l][rows, d:]
        for got, ref, name in ((got_k, k_ref, "K"), (got_v, v_ref, "V")):
            bad = np.abs(got - ref) > 2.0 ** -8 * np.abs(ref) + 1e-3
            assert not bad.any(), f"{what} layer {l} {name}: {bad.sum()} outside the bf16 GEMM bound"
        # against the unrounded memory: add the operand rounding bound
        k_ex, v_ex = R.cross_kv(mem[rows], lw["wk"], lw["wv"], lw["bv"])
        mag_k = np.abs(mem[rows]).astype(np.float64) @ np.abs(lw["wk"]).T.astype(np.float64)
        mag_v = np.abs(mem[rows]).astype(np.float64) @ np.abs(lw["wv"]).T.astype(np.float64)
        assert np.all(np.abs(got_k - k_ex) <= 2.0 ** -8 * np.abs(k_ex) + 2.0 ** -9 * mag_k + 1e-3), f"{what} K"
        assert np.all(np.abs(got_v - v_ex) <= 2.0 ** -8 * np.abs(v_ex) + 2.0 ** -9 * mag_v + 1e-3), f"{what} V"


@pytest.mark.parametrize("cfg_idx,batch,n_ctx,n_layer", [(1, 2, 1500, 4), (1, 1, 37, 2), (4, 1, 300, 2),
                                                         (2, 3, 700, 1)])
def test_prepare_cross_parity(cfg_idx, batch, n_ctx, n_layer):
    cfg = configs.CONFIGS[cfg_idx]
    layers = synth.cross_weights(cfg, n_layer)
    rng = np.random.default_rng(batch * 100 + n_ctx)
    mem = rng.standard_normal((batch, n_ctx, cfg.d_model)).astype(np.float32)
    ckv = wh.CrossKV(cfg.d_model, layers)
    kv = ckv.wh_prepare_cross(torch.from_numpy(mem).cuda())
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    kv = kv.float().cpu().numpy()
    assert kv.shape == (n_layer, batch * n_ctx, 2 * cfg.d_model)
    rows = np.arange(batch * n_ctx)
    _check_cross(kv, mem.reshape(-1, cfg.d_model), layers, rows, cfg.name)


def test_prepare_cross_without_bias():
    cfg = configs.CONFIGS[1]
    layers = synth.cross_weights(cfg, 1)
    layers[0]["bv"] = None
    mem = np.random.default_rng(8).standard_normal((1, 64, cfg.d_model)).astype(np.float32)
    kv = wh.CrossKV(cfg.d_model, layers).wh_prepare_cross(torch.from_numpy(mem).cuda()).float().cpu().numpy()
    _check_cross(kv, mem.reshape(-1, cfg.d_model), layers, np.arange(64), "no bias")


def test_prepare_cross_large_v3_decoder_sampled_rows():
    """The large-v3 decoder's 32 layers over 16 windows (the bench's launch configuration),
    checked on 96 sampled rows of 3 layers (first, a middle one, last)."""
    cfg = configs.CONFIGS[4]
    layers = synth.cross_weights(cfg)
    mem = np.random.default_rng(11).standard_normal((cfg.batch, 1500, cfg.d_model)).astype(np.float32)
    ckv = wh.CrossKV(cfg.d_model, layers)
    kv_d = ckv.wh_prepare_cross(torch.from_numpy(mem).cuda())
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    rows = np.sort(np.random.default_rng(12).choice(cfg.batch * 1500, 96, replace=False))
    rows[-1] = cfg.batch * 1500 - 1
    pick = [0, 17, 31]
    kv = kv_d[pick][:, torch.from_numpy(rows).cuda()].float().cpu().numpy()
    full = np.zeros((len(pick), cfg.batch * 1500, 2 * cfg.d_model), np.float32)
    full[:, rows] = kv
    _check_cross(full, mem.reshape(-1, cfg.d_model), [layers[i] for i in pick], rows, "large-v3")


@pytest.mark.parametrize("cfg_idx", [0, 1])
def test_encode_ctx_full_context_is_wh_encode(cfg_idx):
    cfg = configs.CONFIGS[cfg_idx]
    enc = wh.Encoder(cfg, synth.weights(cfg))
    mel = wh.wh_frontend(torch.from_numpy(synth.waveforms(cfg)).cuda(), cfg.n_mels)
    a = enc.wh_encode(mel)
    b = enc.wh_encode_ctx(mel, 1500)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("cfg_idx,n_ctx,windows", [(1, 500, [0, 5]), (1, 37, [0]), (2, 501, [3]),
                                                   (4, 500, [0])])
def test_encode_ctx_parity(cfg_idx, n_ctx, windows):
    cfg = configs.CONFIGS[cfg_idx]
    w = synth.weights(cfg)
    enc = wh.Encoder(cfg, w)
    pcm = synth.waveforms(cfg)
    mel_d = wh.wh_frontend(torch.from_numpy(pcm).cuda(), cfg.n_mels)
    out = enc.wh_encode_ctx(mel_d, n_ctx)
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    out = out.cpu().numpy()
    mel = mel_d.cpu().numpy()
    assert out.shape == (cfg.batch, n_ctx, cfg.d_model) and np.isfinite(out).all()
    for win in windows:
        ref = R.encoder_ctx(mel[win], w, cfg.n_head, n_ctx)
        check_encoder(out[win], ref, f"{cfg.name} n_ctx {n_ctx} window {win}")


def test_encode_ctx_ignores_frames_past_its_span():
    cfg = configs.CONFIGS[1]
    enc = wh.Encoder(cfg, synth.weights(cfg))
    mel = wh.wh_frontend(torch.from_numpy(synth.waveforms(cfg)).cuda(), cfg.n_mels)
    a = enc.wh_encode_ctx(mel, 400).clone()
    mel[:, 800:] = torch.randn_like(mel[:, 800:])
    b = enc.wh_encode_ctx(mel, 400)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# ---- one-query attention of a decoder step --------------------------------------------------
def _check_attend(out, q, k_rows, v_rows, n_head, what):
    """out bf16 result (numpy float32) of one sequence; q, k_rows, v_rows float32 (bf16 values)."""
    ref = R.attend_one(q, k_rows, v_rows, n_head)
    vmax = float(np.max(np.abs(v_rows))) if v_rows.size else 0.0
    bad = np.abs(out - ref) > 2.0 ** -8 * np.abs(ref) + 1e-4 * max(vmax, 1.0)
    assert not bad.any(), f"{what}: {bad.sum()} outside, max {np.max(np.abs(out - ref)):.3e}"


@pytest.mark.parametrize("batch,n_head,n_keys", [(1, 6, 1500), (3, 8, 37), (2, 20, 1500), (1, 1, 1), (2, 4, 20000)])
def test_decode_attention_dense_cache(batch, n_head, n_keys):
    """K and V as separate [batch][n_keys][64 n_head] caches, every sequence full."""
    rng = np.random.default_rng(batch * 7 + n_head + n_keys)
    D = 64 * n_head
    q = bf16_round_np(rng.standard_normal((batch, D)))
    k = bf16_round_np(rng.standard_normal((batch, n_keys, D)))
    v = bf16_round_np(rng.standard_normal((batch, n_keys, D)))
    dev = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    out = wh.wh_decode_attention(dev(q), dev(k), dev(v), D, n_keys * D, n_keys, n_head)
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    out = out.float().cpu().numpy()
    for b in range(batch):
        _check_attend(out[b], q[b], k[b], v[b], n_head, f"sequence {b}")


def test_decode_attention_over_prepare_cross_rows():
    """The cross-attention of one decoder layer straight off wh_prepare_cross's [K | V] rows."""
    cfg = configs.CONFIGS[1]
    d, H = cfg.d_model, cfg.n_head
    layers = synth.cross_weights(cfg, 2)
    rng = np.random.default_rng(30)
    mem = rng.standard_normal((3, 1500, d)).astype(np.float32)
    kv = wh.CrossKV(d, layers).wh_prepare_cross(torch.from_numpy(mem).cuda())
    q = bf16_round_np(rng.standard_normal((3, d)))
    l = 1
    kl = kv[l]                                        # [3 * 1500][2 d]
    out = wh.wh_decode_attention(torch.from_numpy(q).to(torch.bfloat16).cuda(), kl, kl[:, d:], 2 * d,
                                 1500 * 2 * d, 1500, H)
    torch.cuda.synchronize()
    out = out.float().cpu().numpy()
    kvn = kl.float().cpu().numpy()
    for b in range(3):
        rows = kvn[b * 1500:(b + 1) * 1500]
        _check_attend(out[b], q[b], rows[:, :d], rows[:, d:], H, f"cross window {b}")


def test_decode_attention_ragged_self_cache():
    """A self-attention cache [batch][448][d] with a different length per sequence (0 included)."""
    n_head, cap = 6, 448
    D = 64 * n_head
    lens = np.array([1, 448, 0, 130, 447], dtype=np.int32)
    rng = np.random.default_rng(31)
    q = bf16_round_np(rng.standard_normal((len(lens), D)))
    k = bf16_round_np(rng.standard_normal((len(lens), cap, D)))
    v = bf16_round_np(rng.standard_normal((len(lens), cap, D)))
    dev = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    out = wh.wh_decode_attention(dev(q), dev(k), dev(v), D, cap * D, cap, n_head,
                                 n_keys=torch.from_numpy(lens).cuda())
    torch.cuda.synchronize()
    out = out.float().cpu().numpy()
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(out[b] == 0.0)
        else:
            _check_attend(out[b], q[b], k[b, :n], v[b, :n], n_head, f"sequence {b} ({n} keys)")


def test_decode_attention_key_counts_out_of_range_report_ebounds():
    """Per-sequence key counts live in device memory, so the kernel checks them: a count
    above max_keys or below 0 is clamped (no row past the cache is read) and WH_EBOUNDS is
    recorded; the result equals the call with the clamped counts, and the status word is
    clear again afterwards."""
    n_head, cap = 4, 200
    D = 64 * n_head
    rng = np.random.default_rng(33)
    dev = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    q = dev(bf16_round_np(rng.standard_normal((3, D))))
    k = dev(bf16_round_np(rng.standard_normal((3, cap, D))))
    v = dev(bf16_round_np(rng.standard_normal((3, cap, D))))
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    bad = torch.tensor([cap + 1000, -7, 50], dtype=torch.int32, device="cuda")
    out = wh.wh_decode_attention(q, k, v, D, cap * D, cap, n_head, n_keys=bad).clone()
    assert wh.wh_status() == wh.WH_EBOUNDS
    assert wh.wh_status() == wh.WH_OK                   # read and cleared
    ok = torch.tensor([cap, 0, 50], dtype=torch.int32, device="cuda")
    ref = wh.wh_decode_attention(q, k, v, D, cap * D, cap, n_head, n_keys=ok)
    assert wh.wh_status() == wh.WH_OK
    assert torch.equal(out, ref)


def test_decode_attention_repeated_calls_reuse_the_workspace():
    """The merge tickets are reset by each call: the same workspace gives the same result."""
    rng = np.random.default_rng(32)
    D, n = 64 * 20, 1500
    q = torch.from_numpy(bf16_round_np(rng.standard_normal((16, D)))).to(torch.bfloat16).cuda()
    k = torch.from_numpy(bf16_round_np(rng.standard_normal((16, n, D)))).to(torch.bfloat16).cuda()
    v = torch.from_numpy(bf16_round_np(rng.standard_normal((16, n, D)))).to(torch.bfloat16).cuda()
    ws = torch.empty(wh.lib().wh_decode_attention_workspace(16, 20, n), dtype=torch.uint8, device="cuda")
    a = wh.wh_decode_attention(q, k, v, D, n * D, n, 20, workspace=ws).clone()
    for _ in range(3):
        b = wh.wh_decode_attention(q, k, v, D, n * D, n, 20, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# ---- upstream front end: resampling and long clips -------------------------------------------
@pytest.mark.parametrize("rate", [44100, 48000, 22050, 8000, 11025, 32000, 16000, 16001])
def test_resample_parity(rate):
    rng = np.random.default_rng(rate + 1)
    n = rate // 3 + 101
    x = rng.standard_normal((2, n)).astype(np.float32)
    y = wh.wh_resample(torch.from_numpy(x).cuda(), rate)
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    y = y.cpu().numpy()
    for b in range(2):
        ref = R.resample_to_16k(x[b], rate)
        assert y[b].shape == ref.shape
        err = float(np.max(np.abs(y[b] - ref)))
        assert err <= 1e-5, f"rate {rate}: max |gpu - oracle| {err:.3e}"


def test_long_clip_frontend_matches_its_windows():
    """A 2.26-window clip: each 30-s window's log-mel equals the oracle's on that window
    (zero-padded), and equals wh_frontend on the zero-padded batch bit for bit."""
    cfg = configs.CONFIGS[2]
    n = 2 * 480000 + 123457
    pcm = np.concatenate([synth.waveform(cfg, i) for i in range(3)])[:n]
    mel_long = wh.wh_frontend_long(torch.from_numpy(pcm).cuda(), cfg.n_mels)
    windows = R.long_clip_windows(pcm)
    mel_batch = wh.wh_frontend(torch.from_numpy(np.stack(windows)).cuda(), cfg.n_mels)
    torch.cuda.synchronize()
    assert wh.wh_status() == wh.WH_OK
    assert mel_long.shape == (3, 3000, cfg.n_mels)
    assert torch.equal(mel_long, mel_batch)
    got = mel_long.cpu().numpy()
    for w in (1, 2):
        ref = R.log_mel(windows[w], cfg.n_mels)
        assert float(np.max(np.abs(got[w] - ref))) <= 1e-3


def test_long_clip_frontend_edge_lengths():
    x = torch.from_numpy(synth.waveform(configs.CONFIGS[0], 0)).cuda()
    assert wh.wh_frontend_long(x[:0].contiguous(), 80).shape[0] == 0
    one = wh.wh_frontend_long(x, 80)                              # exactly 480000 samples
    ref = wh.wh_frontend(x[None].contiguous(), 80)
    torch.cuda.synchronize()
    assert one.shape[0] == 1 and torch.equal(one, ref)
