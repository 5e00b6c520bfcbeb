"""The C-ABI library loads, exports every symbol include/wh.h declares, and rejects bad
arguments on the host before touching a device (no compute call is made here)."""
import ctypes
import os
import re

import pytest
import torch

from whisper_audio_encoder_gb300 import build, wh

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wh.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return wh.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wh_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("wh_frontend", "wh_frontend_workspace", "wh_encode", "wh_encode_workspace", "wh_status",
                 "wh_strerror"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing


def test_strerror_names_every_code(L):
    for code in range(7):
        assert wh.wh_strerror(code).startswith("WH_")
    assert "unknown" in wh.wh_strerror(99)


def test_workspace_sizes(L):
    cfg = wh.wh_config(80, 384, 6, 4, 1536)
    one = L.wh_encode_workspace(ctypes.byref(cfg), 1)
    assert one > 0 and L.wh_encode_workspace(ctypes.byref(cfg), 8) > 7 * one
    assert L.wh_frontend_workspace(0) == 0 and L.wh_frontend_workspace(5) >= 20
    bad = wh.wh_config(81, 384, 6, 4, 1536)
    assert L.wh_encode_workspace(ctypes.byref(bad), 1) == 0


FAKE = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("cfg", [(81, 384, 6, 1, 1536), (80, 384, 5, 1, 1536), (80, 320, 5, 1, 1280),
                                 (80, 384, 6, -1, 1536), (80, 384, 6, 1, 100), (128, 4096, 64, 1, 4096)])
def test_encode_rejects_unsupported_configs(L, cfg):
    c = wh.wh_config(*cfg)
    w = wh.wh_weights()
    assert L.wh_encode(FAKE, 1, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL


def test_encode_rejects_null_weights_and_small_workspace(L):
    c = wh.wh_config(80, 384, 6, 0, 1536)
    w = wh.wh_weights()                                   # all NULL
    assert L.wh_encode(FAKE, 1, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL
    assert L.wh_encode(None, 1, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL
    w = wh.wh_weights(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE)
    assert L.wh_encode(FAKE, 1, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 16, None) == wh.WH_ENOSPC
    c.n_layer = 1                                           # layers array missing
    assert L.wh_encode(FAKE, 1, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL
    assert L.wh_encode(FAKE, 0, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 0, None) == wh.WH_OK  # batch 0


def test_encode_rejects_misaligned_pointers(L):
    c = wh.wh_config(80, 384, 6, 0, 1536)
    w = wh.wh_weights(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE)
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert L.wh_encode(odd, 1, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL
    w.pos = odd
    assert L.wh_encode(FAKE, 1, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL


def test_frontend_rejects_bad_arguments(L):
    assert L.wh_frontend(FAKE, 480000, 1, 81, FAKE, FAKE, 256, None) == wh.WH_EINVAL
    assert L.wh_frontend(FAKE, -1, 1, 80, FAKE, FAKE, 256, None) == wh.WH_EINVAL
    assert L.wh_frontend(FAKE, 480000, -1, 80, FAKE, FAKE, 256, None) == wh.WH_EINVAL
    assert L.wh_frontend(FAKE, 480000, 65536, 80, FAKE, FAKE, 1 << 30, None) == wh.WH_EINVAL
    assert L.wh_frontend(None, 480000, 1, 80, FAKE, FAKE, 256, None) == wh.WH_EINVAL
    assert L.wh_frontend(FAKE, 480000, 1, 80, None, FAKE, 256, None) == wh.WH_EINVAL
    assert L.wh_frontend(FAKE, 480000, 1, 80, FAKE, None, 256, None) == wh.WH_EINVAL
    assert L.wh_frontend(FAKE, 480000, 100, 80, FAKE, FAKE, 16, None) == wh.WH_ENOSPC
    assert L.wh_frontend(None, 480000, 0, 80, None, None, 0, None) == wh.WH_OK          # batch 0


def test_single_step_entry_points_reject_bad_shapes(L):
    assert L.wh_layer_norm(FAKE, 4, 100, FAKE, FAKE, FAKE, 1, None) == wh.WH_EINVAL   # d % 64
    assert L.wh_layer_norm(FAKE, 4, 4096, FAKE, FAKE, FAKE, 1, None) == wh.WH_EINVAL  # d > 2048
    assert L.wh_linear(FAKE, 4, 60, FAKE, 128, None, 0, FAKE, None) == wh.WH_EINVAL    # k % 8
    assert L.wh_linear(FAKE, 4, 64, FAKE, 100, None, 0, FAKE, None) == wh.WH_EINVAL    # n % 128
    assert L.wh_linear(FAKE, 4, 64, FAKE, 128, None, 7, FAKE, None) == wh.WH_EINVAL    # epilogue
    assert L.wh_attention(FAKE, 1, 1501, 6, FAKE, None) == wh.WH_EINVAL                # n_ctx > 1500
    assert L.wh_attention(FAKE, 1, 0, 6, FAKE, None) == wh.WH_EINVAL
    assert L.wh_selftest_timeout(0, None) == wh.WH_EINVAL
    assert L.wh_selftest_timeout(2_000_000_000, None) == wh.WH_EINVAL


def test_graph_entry_points_reject_bad_arguments(L):
    c = wh.wh_config(80, 384, 6, 0, 1536)
    w = wh.wh_weights()
    h = ctypes.c_void_p()
    assert L.wh_graph_capture(FAKE, 480000, 1, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, FAKE, 256, FAKE,
                              1 << 30, None, ctypes.byref(h)) == wh.WH_EINVAL          # default stream
    assert L.wh_graph_capture(FAKE, 480000, 1, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, FAKE, 256, FAKE,
                              1 << 30, FAKE, None) == wh.WH_EINVAL                     # no graph slot
    assert L.wh_graph_capture_encode(FAKE, 1, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 1 << 30, None,
                                     ctypes.byref(h)) == wh.WH_EINVAL                  # default stream
    assert L.wh_graph_capture_encode(FAKE, 0, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 1 << 30, FAKE,
                                     ctypes.byref(h)) == wh.WH_EINVAL                  # empty batch
    assert L.wh_graph_launch(None, None) == wh.WH_EINVAL
    assert L.wh_graph_destroy(None) == wh.WH_EINVAL


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_no_device_is_reported(L):
    assert L.wh_frontend(FAKE, 480000, 1, 80, FAKE, FAKE, 256, None) == wh.WH_ENODEV
    assert L.wh_status(None) == wh.WH_ENODEV


def test_encode_ctx_rejects_bad_context(L):
    c = wh.wh_config(80, 384, 6, 0, 1536)
    w = wh.wh_weights(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE)
    for n_ctx in (0, -1, 1501):
        assert L.wh_encode_ctx(FAKE, 1, n_ctx, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 1 << 40, None) \
            == wh.WH_EINVAL
        assert L.wh_encode_ctx_workspace(ctypes.byref(c), 1, n_ctx) == 0
    assert L.wh_encode_ctx(FAKE, 1, 500, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 16, None) == wh.WH_ENOSPC
    assert L.wh_encode_ctx(FAKE, 0, 500, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, 0, None) == wh.WH_OK
    full = L.wh_encode_workspace(ctypes.byref(c), 2)
    assert L.wh_encode_ctx_workspace(ctypes.byref(c), 2, 1500) == full
    assert 0 < L.wh_encode_ctx_workspace(ctypes.byref(c), 2, 500) < full


def test_prepare_cross_rejects_bad_arguments(L):
    ptrs = (ctypes.c_void_p * 2)(FAKE.value, FAKE.value)
    nulls = (ctypes.c_void_p * 2)(None, None)
    cw = wh.wh_cross_weights(ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)),
                             ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)),
                             ctypes.cast(nulls, ctypes.POINTER(ctypes.c_void_p)))
    ok_ws = L.wh_prepare_cross_workspace(2, 1500, 384)
    assert ok_ws >= 2 * 1500 * 384 * 2
    for (d, n_ctx) in ((100, 1500), (384, 0), (384, 1501), (4096, 10), (64, 10)):
        assert L.wh_prepare_cross(FAKE, 2, n_ctx, d, 2, ctypes.byref(cw), FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL
        assert L.wh_prepare_cross_workspace(2, n_ctx, d) == 0
    assert L.wh_prepare_cross(FAKE, 2, 1500, 384, 2, None, FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL
    assert L.wh_prepare_cross(None, 2, 1500, 384, 2, ctypes.byref(cw), FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert L.wh_prepare_cross(odd, 2, 1500, 384, 2, ctypes.byref(cw), FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL
    bad_w = (ctypes.c_void_p * 2)(FAKE.value, None)                 # layer 1's wk missing
    cw_bad = wh.wh_cross_weights(ctypes.cast(bad_w, ctypes.POINTER(ctypes.c_void_p)),
                                 ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)),
                                 ctypes.cast(nulls, ctypes.POINTER(ctypes.c_void_p)))
    assert L.wh_prepare_cross(FAKE, 2, 1500, 384, 2, ctypes.byref(cw_bad), FAKE, FAKE, 1 << 40, None) == wh.WH_EINVAL
    assert L.wh_prepare_cross(FAKE, 2, 1500, 384, 2, ctypes.byref(cw), FAKE, FAKE, 16, None) == wh.WH_ENOSPC
    assert L.wh_prepare_cross(FAKE, 0, 1500, 384, 2, ctypes.byref(cw), FAKE, FAKE, 0, None) == wh.WH_OK
    assert L.wh_prepare_cross(FAKE, 2, 1500, 384, 0, ctypes.byref(cw), FAKE, FAKE, 0, None) == wh.WH_OK


def test_decode_attention_rejects_bad_arguments(L):
    ws = 1 << 30
    assert L.wh_decode_attention_workspace(2, 6, 1500) > 2 * 6 * 66 * 4
    good = (FAKE, FAKE, FAKE, 384, 384 * 1500, None, 1500, 2, 6, FAKE, FAKE, ws, None)
    bad = [dict(i=3, x=100),            # row stride below 64 n_head
           dict(i=3, x=388),            # row stride not a multiple of 8
           dict(i=4, x=-8),             # negative sequence stride
           dict(i=4, x=12),             # sequence stride not a multiple of 8
           dict(i=6, x=0),              # no keys at all
           dict(i=7, x=-1), dict(i=7, x=70000), dict(i=8, x=0),
           dict(i=0, x=None), dict(i=9, x=None),
           dict(i=1, x=ctypes.c_void_p((1 << 20) + 4))]
    for case in bad:
        args = list(good)
        args[case["i"]] = case["x"]
        assert L.wh_decode_attention(*args) == wh.WH_EINVAL, case
    args = list(good)
    args[11] = 64
    assert L.wh_decode_attention(*args) == wh.WH_ENOSPC
    args = list(good)
    args[7] = 0
    assert L.wh_decode_attention(*args) == wh.WH_OK


def test_long_clip_and_resample_argument_checks(L):
    assert L.wh_frontend_windows(0) == 0 and L.wh_frontend_windows(1) == 1
    assert L.wh_frontend_windows(480000) == 1 and L.wh_frontend_windows(480001) == 2
    assert L.wh_frontend_long(FAKE, -1, 80, FAKE, FAKE, 1 << 20, None) == wh.WH_EINVAL
    assert L.wh_frontend_long(FAKE, 480000, 81, FAKE, FAKE, 1 << 20, None) == wh.WH_EINVAL
    assert L.wh_frontend_long(None, 480000, 80, FAKE, FAKE, 1 << 20, None) == wh.WH_EINVAL
    assert L.wh_frontend_long(FAKE, 480000 * 70000, 80, FAKE, FAKE, 1 << 30, None) == wh.WH_EINVAL
    assert L.wh_frontend_long(FAKE, 3 * 480000, 80, FAKE, FAKE, 4, None) == wh.WH_ENOSPC
    assert L.wh_frontend_long(None, 0, 80, None, None, 0, None) == wh.WH_OK
    assert L.wh_resample_length(44100, 44100) == 16000
    assert L.wh_resample_length(1, 44100) == 1 and L.wh_resample_length(0, 8000) == 0
    assert L.wh_resample_length(100, 999) == -1 and L.wh_resample_length(-1, 8000) == -1
    assert L.wh_resample_workspace(999) == 0 and L.wh_resample_workspace(44100) >= 160 * 56 * 4
    assert L.wh_resample(FAKE, 100, 1, 500, FAKE, FAKE, 1 << 20, None) == wh.WH_EINVAL
    assert L.wh_resample(None, 100, 1, 44100, FAKE, FAKE, 1 << 20, None) == wh.WH_EINVAL
    assert L.wh_resample(FAKE, 100, 1, 44100, FAKE, FAKE, 16, None) == wh.WH_ENOSPC
    assert L.wh_resample(FAKE, 0, 1, 44100, FAKE, FAKE, 0, None) == wh.WH_OK


def test_shutdown_forgets_state_and_the_library_sets_up_again(L):
    assert L.wh_shutdown() == wh.WH_OK
    assert L.wh_shutdown() == wh.WH_OK                       # idempotent
    if not torch.cuda.is_available():
        assert L.wh_frontend(FAKE, 480000, 1, 80, FAKE, FAKE, 256, None) == wh.WH_ENODEV


def _dec_cfg(d=384, h=6, layers=1, ff=1536, vocab=1000, ctx=32):
    return wh.wh_dec_config(d, h, layers, ff, vocab, ctx)


@pytest.mark.parametrize("cfg", [(320, 5, 1, 1280, 100, 8), (384, 5, 1, 1536, 100, 8), (384, 6, -1, 1536, 100, 8),
                                 (384, 6, 1, 100, 100, 8), (384, 6, 1, 1536, 0, 8), (384, 6, 1, 1536, 100, 0),
                                 (4096, 64, 1, 4096, 100, 8)])
def test_decode_step_rejects_unsupported_configs(L, cfg):
    c = wh.wh_dec_config(*cfg)
    w = wh.wh_dec_weights()
    assert L.wh_decode_step_workspace(ctypes.byref(c), 4) == 0
    assert L.wh_decode_step(FAKE, FAKE, 4, ctypes.byref(c), ctypes.byref(w), FAKE, FAKE, FAKE, 1500, FAKE, FAKE,
                            FAKE, 1 << 40, None) == wh.WH_EINVAL


def test_decode_step_rejects_bad_arguments_on_the_host(L):
    c = _dec_cfg(layers=0)
    w = wh.wh_dec_weights(FAKE, FAKE, None, FAKE, FAKE)
    call = lambda batch=4, n_ctx=1500, tok=FAKE, ws=1 << 40, wp=w: L.wh_decode_step(
        tok, FAKE, batch, ctypes.byref(c), ctypes.byref(wp), FAKE, FAKE, FAKE, n_ctx, FAKE, FAKE, FAKE, ws, None)
    assert call(batch=0) == wh.WH_OK                                    # no-op
    assert call(batch=257) == wh.WH_EINVAL                              # more sequences than one N tile
    assert call(n_ctx=0) == wh.WH_EINVAL and call(n_ctx=1501) == wh.WH_EINVAL
    assert call(tok=None) == wh.WH_EINVAL
    assert call(tok=ctypes.c_void_p((1 << 20) + 2)) == wh.WH_EINVAL     # misaligned
    assert call(wp=wh.wh_dec_weights()) == wh.WH_EINVAL                 # null weights
    need = L.wh_decode_step_workspace(ctypes.byref(c), 4)
    assert need > 0 and L.wh_decode_step_workspace(ctypes.byref(c), 257) == 0
    assert call(ws=need - 1) == wh.WH_ENOSPC
    c1 = _dec_cfg(layers=1)
    assert L.wh_decode_step(FAKE, FAKE, 4, ctypes.byref(c1), ctypes.byref(w), FAKE, FAKE, FAKE, 1500, FAKE, FAKE,
                            FAKE, 1 << 40, None) == wh.WH_EINVAL               # layers array missing
