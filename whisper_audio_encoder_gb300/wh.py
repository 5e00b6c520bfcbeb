"""Python binding of libwh.so (include/wh.h): argument marshalling only.

Every step of the path runs in the library's CUDA kernels; torch supplies device memory
and streams.  There is no fallback: if libwh.so has not been built, or there is no GPU,
calls raise.
"""
import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libwh.so")

WH_OK, WH_EINVAL, WH_ENOSPC, WH_ECUDA, WH_ETIMEOUT, WH_EBOUNDS, WH_ENODEV = range(7)
WH_EPI_BF16, WH_EPI_GELU_BF16, WH_EPI_RESID_F32 = range(3)
N_CTX, N_FRAMES, N_SAMPLES = 1500, 3000, 480_000

_p = ctypes.c_void_p


class wh_config(ctypes.Structure):
    _fields_ = [("n_mels", ctypes.c_int), ("d_model", ctypes.c_int), ("n_head", ctypes.c_int),
                ("n_layer", ctypes.c_int), ("d_ff", ctypes.c_int)]


class wh_layer_weights(ctypes.Structure):
    _fields_ = [("ln1_g", _p), ("ln1_b", _p), ("wq", _p), ("wk", _p), ("wv", _p), ("bq", _p), ("bv", _p),
                ("wo", _p), ("bo", _p), ("ln2_g", _p), ("ln2_b", _p), ("w1", _p), ("b1", _p),
                ("w2", _p), ("b2", _p)]


class wh_weights(ctypes.Structure):
    _fields_ = [("conv1_w", _p), ("conv1_b", _p), ("conv2_w", _p), ("conv2_b", _p), ("pos", _p),
                ("layers", ctypes.POINTER(wh_layer_weights)), ("lnf_g", _p), ("lnf_b", _p)]


class wh_cross_weights(ctypes.Structure):
    _fields_ = [("wk", ctypes.POINTER(_p)), ("wv", ctypes.POINTER(_p)), ("bv", ctypes.POINTER(_p))]


class wh_dec_config(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("n_head", ctypes.c_int), ("n_layer", ctypes.c_int),
                ("d_ff", ctypes.c_int), ("n_vocab", ctypes.c_int), ("n_text_ctx", ctypes.c_int)]


_DEC_LAYER_FIELDS = ["ln1_g", "ln1_b", "wq", "wk", "wv", "bq", "bv", "wo", "bo", "lnx_g", "lnx_b", "xwq", "xbq",
                     "xwo", "xbo", "ln2_g", "ln2_b", "w1", "b1", "w2", "b2"]


class wh_dec_layer_weights(ctypes.Structure):
    _fields_ = [(n, _p) for n in _DEC_LAYER_FIELDS]


class wh_dec_weights(ctypes.Structure):
    _fields_ = [("tok_embd", _p), ("pos", _p), ("layers", ctypes.POINTER(wh_dec_layer_weights)),
                ("lnf_g", _p), ("lnf_b", _p)]


class wh_trace_stat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


class WhError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {wh_strerror(code)}" if what else wh_strerror(code))


_lib = None


def lib():
    """Loads libwh.so (built in-tree by whisper_audio_encoder_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m whisper_audio_encoder_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(LIB_PATH)
    sig = {
        "wh_frontend_workspace": (ctypes.c_size_t, [ctypes.c_int]),
        "wh_frontend": (ctypes.c_int, [_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _p, _p, ctypes.c_size_t, _p]),
        "wh_frontend_static": (ctypes.c_int, [_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _p, _p]),
        "wh_encode_workspace": (ctypes.c_size_t, [ctypes.POINTER(wh_config), ctypes.c_int]),
        "wh_encode": (ctypes.c_int, [_p, ctypes.c_int, ctypes.POINTER(wh_config), ctypes.POINTER(wh_weights),
                                     _p, _p, ctypes.c_size_t, _p]),
        "wh_encode_ctx_workspace": (ctypes.c_size_t, [ctypes.POINTER(wh_config), ctypes.c_int, ctypes.c_int]),
        "wh_encode_ctx": (ctypes.c_int, [_p, ctypes.c_int, ctypes.c_int, ctypes.POINTER(wh_config),
                                         ctypes.POINTER(wh_weights), _p, _p, ctypes.c_size_t, _p]),
        "wh_prepare_cross_workspace": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
        "wh_prepare_cross": (ctypes.c_int, [_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.POINTER(wh_cross_weights), _p, _p, ctypes.c_size_t, _p]),
        "wh_decode_attention_workspace": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
        "wh_decode_attention": (ctypes.c_int, [_p, _p, _p, ctypes.c_int64, ctypes.c_int64, _p, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, _p, _p, ctypes.c_size_t, _p]),
        "wh_decode_step_workspace": (ctypes.c_size_t, [ctypes.POINTER(wh_dec_config), ctypes.c_int]),
        "wh_decode_step": (ctypes.c_int, [_p, _p, ctypes.c_int, ctypes.POINTER(wh_dec_config),
                                          ctypes.POINTER(wh_dec_weights), _p, _p, _p, ctypes.c_int, _p, _p, _p,
                                          ctypes.c_size_t, _p]),
        "wh_frontend_windows": (ctypes.c_int64, [ctypes.c_int64]),
        "wh_frontend_long": (ctypes.c_int, [_p, ctypes.c_int64, ctypes.c_int, _p, _p, ctypes.c_size_t, _p]),
        "wh_resample_length": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int]),
        "wh_resample_workspace": (ctypes.c_size_t, [ctypes.c_int]),
        "wh_resample": (ctypes.c_int, [_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _p, _p, ctypes.c_size_t, _p]),
        "wh_layer_norm": (ctypes.c_int, [_p, ctypes.c_int, ctypes.c_int, _p, _p, _p, ctypes.c_int, _p]),
        "wh_linear": (ctypes.c_int, [_p, ctypes.c_int, ctypes.c_int, _p, ctypes.c_int, _p, ctypes.c_int, _p, _p]),
        "wh_attention": (ctypes.c_int, [_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _p, _p]),
        "wh_status": (ctypes.c_int, [_p]),
        "wh_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "wh_shutdown": (ctypes.c_int, []),
        "wh_selftest_timeout": (ctypes.c_int, [ctypes.c_uint64, _p]),
        "wh_trace_enable": (ctypes.c_int, [ctypes.c_int]),
        "wh_trace_read": (ctypes.c_int, [ctypes.POINTER(wh_trace_stat), ctypes.c_int]),
        "wh_launch_count": (ctypes.c_int64, []),
        "wh_graph_capture": (ctypes.c_int, [_p, ctypes.c_int64, ctypes.c_int, ctypes.POINTER(wh_config),
                                            ctypes.POINTER(wh_weights), _p, _p, _p, ctypes.c_size_t, _p,
                                            ctypes.c_size_t, _p, ctypes.POINTER(ctypes.c_void_p)]),
        "wh_graph_capture_encode": (ctypes.c_int, [_p, ctypes.c_int, ctypes.POINTER(wh_config),
                                                   ctypes.POINTER(wh_weights), _p, _p, ctypes.c_size_t, _p,
                                                   ctypes.POINTER(ctypes.c_void_p)]),
        "wh_graph_capture_decode": (ctypes.c_int, [_p, _p, ctypes.c_int, ctypes.POINTER(wh_dec_config),
                                                   ctypes.POINTER(wh_dec_weights), _p, _p, _p, ctypes.c_int, _p, _p,
                                                   _p, ctypes.c_size_t, _p, ctypes.POINTER(ctypes.c_void_p)]),
        "wh_graph_launch": (ctypes.c_int, [_p, _p]),
        "wh_graph_destroy": (ctypes.c_int, [_p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def wh_strerror(code: int) -> str:
    return lib().wh_strerror(code).decode()


def _check(rc, what):
    if rc != WH_OK:
        raise WhError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ---------------------------------------------------------------------------------------
# Entry points (same names as the C ABI), taking torch tensors
# ---------------------------------------------------------------------------------------
def wh_frontend_workspace(batch: int) -> int:
    return lib().wh_frontend_workspace(batch)


def wh_frontend(pcm, n_mels: int, mel=None, workspace=None, stream=None):
    """pcm: float32 CUDA tensor [batch][n] -> log-mel float32 [batch][3000][n_mels]."""
    import torch
    assert pcm.dtype == torch.float32 and pcm.dim() == 2 and pcm.is_contiguous()
    batch, n = pcm.shape
    if mel is None:
        mel = torch.empty(batch, N_FRAMES, n_mels, dtype=torch.float32, device=pcm.device)
    if workspace is None:
        workspace = torch.empty(max(16, wh_frontend_workspace(batch)), dtype=torch.uint8, device=pcm.device)
    rc = lib().wh_frontend(_ptr(pcm), n, batch, n_mels, _ptr(mel), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    _check(rc, "wh_frontend")
    return mel


def wh_frontend_long(pcm, n_mels: int, mel=None, workspace=None, stream=None):
    """One long clip, float32 CUDA tensor [n] -> log-mel [ceil(n / 480000)][3000][n_mels]
    (consecutive 30-s windows, the last zero-padded)."""
    import torch
    assert pcm.dtype == torch.float32 and pcm.dim() == 1 and pcm.is_contiguous()
    n = pcm.shape[0]
    windows = lib().wh_frontend_windows(n)
    if mel is None:
        mel = torch.empty(max(windows, 0), N_FRAMES, n_mels, dtype=torch.float32, device=pcm.device)
    if workspace is None:
        workspace = torch.empty(max(16, wh_frontend_workspace(max(windows, 1))), dtype=torch.uint8, device=pcm.device)
    _check(lib().wh_frontend_long(_ptr(pcm), n, n_mels, _ptr(mel), _ptr(workspace), workspace.numel(),
                                  _stream(stream)), "wh_frontend_long")
    return mel


def wh_resample(x, rate_in: int, y=None, workspace=None, stream=None):
    """x float32 CUDA tensor [batch][n] at rate_in Hz -> [batch][n_out] at 16 kHz."""
    import torch
    assert x.dtype == torch.float32 and x.dim() == 2 and x.is_contiguous()
    batch, n = x.shape
    n_out = lib().wh_resample_length(n, rate_in)
    if n_out < 0:
        raise WhError(WH_EINVAL, "wh_resample_length")
    if y is None:
        y = torch.empty(batch, n_out, dtype=torch.float32, device=x.device)
    need = max(256, lib().wh_resample_workspace(rate_in))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _check(lib().wh_resample(_ptr(x), n, batch, rate_in, _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)),
           "wh_resample")
    return y


def wh_layer_norm(x, g, b, out_bf16=True, y=None, stream=None):
    import torch
    rows, d = x.shape
    if y is None:
        y = torch.empty(rows, d, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=x.device)
    _check(lib().wh_layer_norm(_ptr(x), rows, d, _ptr(g), _ptr(b), _ptr(y), int(out_bf16), _stream(stream)),
           "wh_layer_norm")
    return y


def wh_linear(a, w, bias=None, epilogue=WH_EPI_BF16, y=None, stream=None):
    """a bf16 [rows][k], w bf16 [n][k] -> y (bf16, or the fp32 residual updated in place)."""
    import torch
    rows, k = a.shape
    n = w.shape[0]
    if y is None:
        y = torch.empty(rows, n, dtype=torch.bfloat16, device=a.device)
    _check(lib().wh_linear(_ptr(a), rows, k, _ptr(w), n, _ptr(bias), epilogue, _ptr(y), _stream(stream)),
           "wh_linear")
    return y


def wh_attention(qkv, batch, n_ctx, n_head, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty(batch * n_ctx, n_head * 64, dtype=torch.bfloat16, device=qkv.device)
    _check(lib().wh_attention(_ptr(qkv), batch, n_ctx, n_head, _ptr(out), _stream(stream)), "wh_attention")
    return out


def wh_decode_attention(q, k, v, row_stride, seq_stride, max_keys, n_head, n_keys=None, out=None,
                        workspace=None, stream=None):
    """One query per (sequence, head) over up to max_keys keys: q bf16 [batch][64 n_head];
    k / v bf16 device tensors (views are fine) addressed with the given element strides;
    n_keys: optional int32 device tensor [batch].  Returns bf16 [batch][64 n_head]."""
    import torch
    batch = q.shape[0]
    if out is None:
        out = torch.empty(batch, 64 * n_head, dtype=torch.bfloat16, device=q.device)
    need = max(256, lib().wh_decode_attention_workspace(batch, n_head, max_keys))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    rc = lib().wh_decode_attention(_ptr(q), _ptr(k), _ptr(v), row_stride, seq_stride, _ptr(n_keys), max_keys, batch,
                                   n_head, _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "wh_decode_attention")
    return out


def wh_status(stream=None) -> int:
    return lib().wh_status(_stream(stream))


def wh_selftest_timeout(limit_ns: int, stream=None):
    _check(lib().wh_selftest_timeout(limit_ns, _stream(stream)), "wh_selftest_timeout")


def wh_launch_count() -> int:
    return lib().wh_launch_count()


def wh_trace_enable(on: bool):
    lib().wh_trace_enable(int(on))


def wh_trace_read():
    arr = (wh_trace_stat * 32)()
    n = lib().wh_trace_read(arr, 32)
    if n < 0:
        raise WhError(-n, "wh_trace_read")
    return {arr[i].name.decode(): {"launches": arr[i].launches, "total_ms": arr[i].total_ms,
                                   "flops": arr[i].flops, "bytes": arr[i].bytes} for i in range(n)}


# ---------------------------------------------------------------------------------------
# Encoder: device weights + the wh_weights struct + workspace
# ---------------------------------------------------------------------------------------
class Encoder:
    """Holds an encoder's weights on the device and calls wh_encode.

    `weights` is a dict of numpy arrays (matrices already bf16-representable float32,
    vectors float32), as produced by whisper_audio_encoder_gb300.synth.weights."""

    def __init__(self, cfg, weights: dict, device="cuda"):
        import torch
        self.cfg = cfg
        self.device = torch.device(device)
        self._keep = []

        def mat(a):
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).to(self.device)
            self._keep.append(t)
            return t.data_ptr()

        def vec(a):
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(self.device)
            self._keep.append(t)
            return t.data_ptr()

        n_layer = len(weights["layers"])
        self.c_cfg = wh_config(cfg.n_mels, cfg.d_model, cfg.n_head, n_layer, cfg.d_ff)
        self._layers = (wh_layer_weights * max(1, n_layer))()
        for i, lw in enumerate(weights["layers"]):
            L = self._layers[i]
            L.ln1_g, L.ln1_b = vec(lw["ln1_g"]), vec(lw["ln1_b"])
            L.wq, L.wk, L.wv = mat(lw["wq"]), mat(lw["wk"]), mat(lw["wv"])
            L.bq, L.bv = vec(lw["bq"]), vec(lw["bv"])
            L.wo, L.bo = mat(lw["wo"]), vec(lw["bo"])
            L.ln2_g, L.ln2_b = vec(lw["ln2_g"]), vec(lw["ln2_b"])
            L.w1, L.b1 = mat(lw["w1"]), vec(lw["b1"])
            L.w2, L.b2 = mat(lw["w2"]), vec(lw["b2"])
        self.c_w = wh_weights(mat(weights["conv1_w"]), vec(weights["conv1_b"]), mat(weights["conv2_w"]),
                              vec(weights["conv2_b"]), vec(weights["pos"]),
                              ctypes.cast(self._layers, ctypes.POINTER(wh_layer_weights)),
                              vec(weights["lnf_g"]), vec(weights["lnf_b"]))
        self._ws = None
        self._fe_ws = None

    def workspace_bytes(self, batch: int, n_ctx: int = N_CTX) -> int:
        return lib().wh_encode_ctx_workspace(ctypes.byref(self.c_cfg), batch, n_ctx)

    def workspace(self, batch: int, n_ctx: int = N_CTX):
        import torch
        need = self.workspace_bytes(batch, n_ctx)
        if self._ws is None or self._ws.numel() < need:
            self._ws = None
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def wh_encode(self, mel, out=None, stream=None):
        """mel float32 [batch][3000][n_mels] (device) -> float32 [batch][1500][d_model]."""
        import torch
        batch = mel.shape[0]
        if out is None:
            out = torch.empty(batch, N_CTX, self.cfg.d_model, dtype=torch.float32, device=self.device)
        ws = self.workspace(batch)
        rc = lib().wh_encode(_ptr(mel), batch, ctypes.byref(self.c_cfg), ctypes.byref(self.c_w), _ptr(out),
                             _ptr(ws), ws.numel(), _stream(stream))
        _check(rc, "wh_encode")
        return out

    def wh_encode_ctx(self, mel, n_ctx: int, out=None, stream=None):
        """The encoder over the first 2 n_ctx frames of each window's log-mel:
        mel float32 [batch][3000][n_mels] (device) -> float32 [batch][n_ctx][d_model]."""
        import torch
        batch = mel.shape[0]
        if out is None:
            out = torch.empty(batch, n_ctx, self.cfg.d_model, dtype=torch.float32, device=self.device)
        ws = self.workspace(batch, n_ctx)
        rc = lib().wh_encode_ctx(_ptr(mel), batch, n_ctx, ctypes.byref(self.c_cfg), ctypes.byref(self.c_w),
                                 _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
        _check(rc, "wh_encode_ctx")
        return out

    def frontend_workspace(self, batch: int):
        import torch
        need = max(16, wh_frontend_workspace(batch))
        if self._fe_ws is None or self._fe_ws.numel() < need:
            self._fe_ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._fe_ws

    def forward(self, pcm, mel=None, out=None, stream=None):
        """16 kHz PCM float32 [batch][n] on the device -> encoder memory [batch][1500][d]."""
        mel = wh_frontend(pcm, self.cfg.n_mels, mel=mel, workspace=self.frontend_workspace(pcm.shape[0]),
                          stream=stream)
        return self.wh_encode(mel, out=out, stream=stream)

    def capture(self, pcm, mel, out, stream):
        """Records one front end + encoder pass over these device buffers (wh_graph_capture).
        `stream` is a torch.cuda.Stream other than the default stream; replay with
        Graph.launch(); refresh `pcm` in place between replays."""
        batch, n = pcm.shape
        ws = self.workspace(batch)
        fe = self.frontend_workspace(batch)
        h = ctypes.c_void_p()
        rc = lib().wh_graph_capture(_ptr(pcm), n, batch, ctypes.byref(self.c_cfg), ctypes.byref(self.c_w), _ptr(mel),
                                    _ptr(out), _ptr(fe), fe.numel(), _ptr(ws), ws.numel(), _stream(stream),
                                    ctypes.byref(h))
        _check(rc, "wh_graph_capture")
        return Graph(h, (pcm, mel, out, ws, fe))

    def capture_encode(self, mel, out, stream):
        """Records one wh_encode pass (mel -> memory) over these device buffers."""
        batch = mel.shape[0]
        ws = self.workspace(batch)
        h = ctypes.c_void_p()
        rc = lib().wh_graph_capture_encode(_ptr(mel), batch, ctypes.byref(self.c_cfg), ctypes.byref(self.c_w), _ptr(out),
                                           _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(h))
        _check(rc, "wh_graph_capture_encode")
        return Graph(h, (mel, out, ws))

    def encode_from_host(self, pcm_host, out_host, pcm_dev, mel, out_dev, stream=None):
        """End to end from pinned host memory: copy PCM in, front end + encoder, copy the
        memory out (all on one stream)."""
        pcm_dev.copy_(pcm_host, non_blocking=True)
        self.forward(pcm_dev, mel=mel, out=out_dev, stream=stream)
        out_host.copy_(out_dev, non_blocking=True)
        return out_host


class Graph:
    """A recorded front end + encoder pass (wh_graph_*); keeps its buffers alive."""

    def __init__(self, handle, keep):
        self._h = handle
        self._keep = keep

    def launch(self, stream=None):
        _check(lib().wh_graph_launch(self._h, _stream(stream)), "wh_graph_launch")

    def destroy(self):
        if self._h:
            lib().wh_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


# ---------------------------------------------------------------------------------------
# Cross-attention K/V of the decoder layers (wh_prepare_cross)
# ---------------------------------------------------------------------------------------
class CrossKV:
    """Holds the decoder layers' cross-attention k/v projections on the device and calls
    wh_prepare_cross.  `layers` is a list of dicts with "wk", "wv" (bf16-representable
    float32 [d][d]) and "bv" (float32 [d] or None)."""

    def __init__(self, d_model: int, layers, device="cuda"):
        import torch
        self.d_model = d_model
        self.n_layer = len(layers)
        self.device = torch.device(device)
        self._keep = []

        def put(a, dtype):
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dtype).to(self.device)
            self._keep.append(t)
            return t.data_ptr()

        n = max(1, self.n_layer)
        self._wk, self._wv, self._bv = (_p * n)(), (_p * n)(), (_p * n)()
        for i, lw in enumerate(layers):
            self._wk[i] = put(lw["wk"], torch.bfloat16)
            self._wv[i] = put(lw["wv"], torch.bfloat16)
            self._bv[i] = None if lw.get("bv") is None else put(lw["bv"], torch.float32)
        self.c_w = wh_cross_weights(ctypes.cast(self._wk, ctypes.POINTER(_p)), ctypes.cast(self._wv, ctypes.POINTER(_p)),
                                    ctypes.cast(self._bv, ctypes.POINTER(_p)))
        self._ws = None

    def wh_prepare_cross(self, mem, kv=None, stream=None):
        """mem float32 [batch][n_ctx][d] (device) -> kv bf16 [n_layer][batch * n_ctx][2 d]:
        K in columns 0..d-1, V in d..2d-1."""
        import torch
        batch, n_ctx, d = mem.shape
        assert d == self.d_model and mem.dtype == torch.float32 and mem.is_contiguous()
        if kv is None:
            kv = torch.empty(self.n_layer, batch * n_ctx, 2 * d, dtype=torch.bfloat16, device=self.device)
        need = max(256, lib().wh_prepare_cross_workspace(batch, n_ctx, d))
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        rc = lib().wh_prepare_cross(_ptr(mem), batch, n_ctx, d, self.n_layer, ctypes.byref(self.c_w), _ptr(kv),
                                    _ptr(self._ws), self._ws.numel(), _stream(stream))
        _check(rc, "wh_prepare_cross")
        return kv


class Pipeline:
    """A double-buffered serving loop over recorded passes.

    Two device buffer sets, each with its own recorded front end + encoder pass (the
    log-mel buffer and the encoder workspace are shared: the passes run one after the other
    on the compute stream).  While batch k is encoded, batch k+1's PCM is copied in on one
    copy stream and batch k-1's encoder memory is copied out on another; stream events keep
    a buffer from being overwritten before the pass or copy that uses it has finished."""

    def __init__(self, enc, batch: int, n_samples: int = N_SAMPLES):
        import torch
        dev = enc.device
        self.enc = enc
        self.compute = torch.cuda.Stream(dev)
        self.copy_in = torch.cuda.Stream(dev)
        self.copy_out = torch.cuda.Stream(dev)
        self.mel = torch.empty(batch, N_FRAMES, enc.cfg.n_mels, dtype=torch.float32, device=dev)
        self.pcm = [torch.empty(batch, n_samples, dtype=torch.float32, device=dev) for _ in range(2)]
        self.out = [torch.empty(batch, N_CTX, enc.cfg.d_model, dtype=torch.float32, device=dev) for _ in range(2)]
        self.graphs = [enc.capture(self.pcm[i], self.mel, self.out[i], self.compute) for i in range(2)]
        self.in_done = [torch.cuda.Event() for _ in range(2)]
        self.pass_done = [torch.cuda.Event() for _ in range(2)]
        self.out_done = [torch.cuda.Event() for _ in range(2)]

    def run(self, pcm_host, out_host):
        """pcm_host / out_host: lists of pinned host tensors, one per batch; encodes them in
        order and returns when every result is on the host."""
        import torch
        for k, (src, dst) in enumerate(zip(pcm_host, out_host)):
            i = k & 1
            self.copy_in.wait_event(self.pass_done[i])        # the pass that read pcm[i] is done
            with torch.cuda.stream(self.copy_in):
                self.pcm[i].copy_(src, non_blocking=True)
            self.in_done[i].record(self.copy_in)
            self.compute.wait_event(self.in_done[i])
            self.compute.wait_event(self.out_done[i])         # out[i] has been copied out
            self.graphs[i].launch(self.compute)
            self.pass_done[i].record(self.compute)
            self.copy_out.wait_event(self.pass_done[i])
            with torch.cuda.stream(self.copy_out):
                dst.copy_(self.out[i], non_blocking=True)
            self.out_done[i].record(self.copy_out)
        self.copy_out.synchronize()

    def destroy(self):
        for g in self.graphs:
            g.destroy()


# ---------------------------------------------------------------------------------------
# Decoder step (wh_decode_step): device weights, self-attention caches, workspace
# ---------------------------------------------------------------------------------------
class Decoder:
    """Holds a decoder's weights and its self-attention caches on the device and calls
    wh_decode_step.  `weights` is a dict as produced by synth.decoder_weights: "tok_embd"
    [n_vocab][d] and matrices bf16-representable float32, vectors float32, "layers" a list of
    per-block dicts.  The caches are bf16 [n_layer][batch][n_text_ctx][d_model]."""

    def __init__(self, n_head: int, weights: dict, batch: int, device="cuda"):
        import torch
        self.device = torch.device(device)
        self._keep = []

        def put(a, dtype):
            if isinstance(a, torch.Tensor):
                t = a.to(device=self.device, dtype=dtype).contiguous()
            else:
                t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dtype).to(self.device)
            self._keep.append(t)
            return t.data_ptr()

        n_vocab, d = weights["tok_embd"].shape
        n_text_ctx = weights["dec_pos"].shape[0]
        n_layer = len(weights["layers"])
        d_ff = weights["layers"][0]["w1"].shape[0] if n_layer else 4 * d
        self.batch = batch
        self.c_cfg = wh_dec_config(d, n_head, n_layer, d_ff, n_vocab, n_text_ctx)
        self._layers = (wh_dec_layer_weights * max(1, n_layer))()
        for i, lw in enumerate(weights["layers"]):
            L = self._layers[i]
            for name in _DEC_LAYER_FIELDS:
                is_mat = name in ("wq", "wk", "wv", "wo", "xwq", "xwo", "w1", "w2")
                setattr(L, name, put(lw[name], torch.bfloat16 if is_mat else torch.float32))
        self.c_w = wh_dec_weights(put(weights["tok_embd"], torch.bfloat16), put(weights["dec_pos"], torch.float32),
                                  ctypes.cast(self._layers, ctypes.POINTER(wh_dec_layer_weights)),
                                  put(weights["lnf_g"], torch.float32), put(weights["lnf_b"], torch.float32))
        shape = (max(1, n_layer), batch, n_text_ctx, d)
        self.kcache = torch.zeros(shape, dtype=torch.bfloat16, device=self.device)
        self.vcache = torch.zeros(shape, dtype=torch.bfloat16, device=self.device)
        self.logits = torch.empty(batch, n_vocab, dtype=torch.float32, device=self.device)
        self.next_tok = torch.empty(batch, dtype=torch.int32, device=self.device)
        need = max(256, lib().wh_decode_step_workspace(ctypes.byref(self.c_cfg), batch))
        self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)

    def wh_decode_step(self, tok, pos, cross_kv, n_ctx: int, stream=None):
        """tok, pos: int32 device tensors [batch]; cross_kv: bf16 [n_layer][batch * n_ctx][2 d]
        (wh_prepare_cross's output).  Returns (logits [batch][n_vocab], next_tok [batch])."""
        import torch
        assert tok.dtype == torch.int32 and pos.dtype == torch.int32 and cross_kv.dtype == torch.bfloat16
        rc = lib().wh_decode_step(_ptr(tok), _ptr(pos), self.batch, ctypes.byref(self.c_cfg), ctypes.byref(self.c_w),
                                  _ptr(self.kcache), _ptr(self.vcache), _ptr(cross_kv), n_ctx, _ptr(self.logits),
                                  _ptr(self.next_tok), _ptr(self.workspace), self.workspace.numel(), _stream(stream))
        _check(rc, "wh_decode_step")
        return self.logits, self.next_tok

    def capture(self, tok, pos, cross_kv, n_ctx: int, stream):
        """Records one wh_decode_step over these buffers (wh_graph_capture_decode); replay with
        Graph.launch() after refreshing tok / pos in place."""
        h = ctypes.c_void_p()
        rc = lib().wh_graph_capture_decode(_ptr(tok), _ptr(pos), self.batch, ctypes.byref(self.c_cfg),
                                           ctypes.byref(self.c_w), _ptr(self.kcache), _ptr(self.vcache),
                                           _ptr(cross_kv), n_ctx, _ptr(self.logits), _ptr(self.next_tok),
                                           _ptr(self.workspace), self.workspace.numel(), _stream(stream),
                                           ctypes.byref(h))
        _check(rc, "wh_graph_capture_decode")
        return Graph(h, (tok, pos, cross_kv))
