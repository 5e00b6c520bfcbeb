"""Plain CPU oracle of the Whisper audio-encoder forward pass.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU-baseline /
reference arm may import this module; the library never does, and this module imports
nothing from the library.  It is deliberately slow and literal: every step is the plain
definition of what the step computes, in float64, with a library primitive (a matrix
product, erf, exp) as the only building block.  No FFT, no blocking, no fusion.

Sources (web pages the method is described on; section names as they appear there):
  [CKE]  "How Audio Becomes Words: Whisper's Kernels Step By Step On A CPU"
         -- section "The Frontend: Sound Becomes A Tensor" (the eight front-end kernels and
            the bullets that walk them), "The Encoder: Understand Once",
            "The Full Stitched Circuit", "Tiny, Base, Small, Large".
  [API]  "whisper 0.9.0 API" -- model.nu (encoder shape, k_proj without bias, wh_encode
         layouts, wh_prepare_cross, wh_decode_step), kernels.nu (LayerNorm with bias, erf
         GELU, conv1d, non-causal attention with the 1/sqrt(hd) score scale) and main.nu
         (long audio in 30-s windows).
  [README] the "whisper" package page -- "Serving" (draft encoder over a shorter context),
         "Transcribing" and "How it is verified" (windowed-sinc resampling to 16 kHz,
         checked against resample_poly), "Performance and memory" (one-query attention with
         the keys split across blocks).

Readings where the pages are silent (each is a decision, recorded with the code):
  r1  3000 frames: centred, reflect-padded frames t = 0..2999 (the 3001st is dropped).
  r2  reflect = mirror without repeating the edge sample (x[-1] = x[1]).
  r3  Hann is periodic: 0.5 - 0.5 cos(2 pi n / 400).
  r4  power = re^2 + im^2.
  r5  Slaney mel scale, M+2 points equally spaced in mel over [0, 8000] Hz, triangles
      area-normalised by 2 / (f[m+2] - f[m]), evaluated at bin frequencies 40 k Hz.
  r6  log floor 1e-10 inside log10.
  r7  the "global" maximum is per window (per 30-s clip).
  r8  clamp at (max - 8) in log10 units, i.e. -80 dB of power.
  r9  conv padding is zeros.
  r10 LayerNorm eps 1e-5, biased variance.
  r11 GELU is the exact erf form.
  r12 scores scaled by 1/sqrt(64); head h owns columns [64 h, 64 h + 64).
  r13 GELU after each conv; positions added after conv2's GELU.
  r20 a shorter encoder context reads the first 2 n_ctx frames and zero-pads at their end.
  r21 the windowed-sinc resampler is resample_poly's default design (Kaiser beta 5, 10 M
      taps on each side, unit DC gain).
  r22 long clips are cut into consecutive, non-overlapping 30-s windows, the last padded.
  r23 a decode step writes the token's own key and value at row pos of the self-attention
      cache first and then attends over rows 0..pos (the cache "holds what came before it";
      the one query at the end attends to itself too, as every causal row does).

Pinned by tests/test_oracle_*.py against closed forms, invariants, library routines
(numpy.fft, torch.stft, torch.nn.functional) and brute force.  The full encoder has no
published value to pin it: it is pinned by an independent restatement with torch CPU ops.
"""
import numpy as np
from scipy.special import erf

SAMPLE_RATE = 16_000
N_SAMPLES = 480_000
N_FFT = 400
HOP = 160
N_FRAMES = 3000
N_BINS = N_FFT // 2 + 1      # 201
N_CTX = 1500
HEAD_DIM = 64
LN_EPS = 1e-5
LOG_FLOOR = 1e-10


# ========================================================================================
# Front end  [CKE] "The Frontend: Sound Becomes A Tensor", kernels 3-6 and their bullets
# ========================================================================================
def pad_or_truncate(pcm: np.ndarray, n_samples: int = N_SAMPLES) -> np.ndarray:
    """Kernel 3 'pad or truncate': zero-pad short clips, cut long ones, to 480000 samples."""
    x = np.zeros(n_samples, dtype=np.float64)
    m = min(len(pcm), n_samples)
    x[:m] = pcm[:m]
    return x


def hann_periodic(n_fft: int = N_FFT) -> np.ndarray:
    """Kernel 4 'periodic Hann' (r3): w[n] = 0.5 - 0.5 cos(2 pi n / N), n = 0..N-1."""
    n = np.arange(n_fft, dtype=np.float64)
    return 0.5 - 0.5 * np.cos(2.0 * np.pi * n / n_fft)


def frame_signal(x: np.ndarray) -> np.ndarray:
    """Kernel 4 'reflect-pad' and framing (r1, r2): frame t holds samples
    160 t - 200 .. 160 t + 199 of x, an index i < 0 reading x[-i] and an index i > N-1
    reading x[2 (N-1) - i].  Returns float64 [3000][400]."""
    n = len(x)
    half = N_FFT // 2
    t = np.arange(N_FRAMES)[:, None]
    j = np.arange(N_FFT)[None, :]
    i = HOP * t + j - half
    i = np.where(i < 0, -i, i)
    i = np.where(i > n - 1, 2 * (n - 1) - i, i)
    return x[i].astype(np.float64)


def dft_power(frames: np.ndarray, window: np.ndarray) -> np.ndarray:
    """Kernel 4 'STFT power' (r4): P[t][k] = |sum_n w[n] frame_t[n] exp(-2 pi i k n / 400)|^2
    for k = 0..200, by the direct definition (a float64 matrix product, no FFT)."""
    n = np.arange(N_FFT, dtype=np.float64)[:, None]
    k = np.arange(N_BINS, dtype=np.float64)[None, :]
    ang = 2.0 * np.pi * ((n * k) % N_FFT) / N_FFT      # reduce n k mod N before the angle
    xw = frames * window[None, :]
    re = xw @ np.cos(ang)
    im = -(xw @ np.sin(ang))
    return re * re + im * im


def hz_to_mel_slaney(f):
    """Slaney mel scale (r5): linear below 1 kHz (3 f / 200), logarithmic above,
    with 27 mel per factor 6.4 in frequency."""
    f = np.asarray(f, dtype=np.float64)
    lin = 3.0 * f / 200.0
    logpart = 15.0 + 27.0 * np.log(np.maximum(f, 1e-300) / 1000.0) / np.log(6.4)
    return np.where(f < 1000.0, lin, logpart)


def mel_to_hz_slaney(m):
    m = np.asarray(m, dtype=np.float64)
    lin = 200.0 * m / 3.0
    logpart = 1000.0 * np.exp((m - 15.0) * np.log(6.4) / 27.0)
    return np.where(m < 15.0, lin, logpart)


def mel_filterbank(n_mels: int, sr: int = SAMPLE_RATE, n_fft: int = N_FFT) -> np.ndarray:
    """Kernel 5 'mel filters': n_mels triangles on the Slaney scale, area-normalised (r5).
    Returns float64 [n_mels][201]."""
    edges_mel = np.linspace(hz_to_mel_slaney(0.0), hz_to_mel_slaney(sr / 2.0), n_mels + 2)
    f = mel_to_hz_slaney(edges_mel)                                 # [n_mels + 2] Hz
    bins = np.arange(n_fft // 2 + 1, dtype=np.float64) * sr / n_fft  # 40 Hz apart
    fb = np.zeros((n_mels, len(bins)))
    for m in range(n_mels):
        lo, c, hi = f[m], f[m + 1], f[m + 2]
        rising = (bins - lo) / (c - lo)
        falling = (hi - bins) / (hi - c)
        fb[m] = np.maximum(0.0, np.minimum(rising, falling)) * (2.0 / (hi - lo))
    return fb


def log_mel_from_power(power: np.ndarray, fb: np.ndarray) -> np.ndarray:
    """Kernels 5-6: mel projection, log10 with floor (r6), clamp at the window maximum
    minus 8 (r7, r8), then (x + 4) / 4.  power [3000][201] -> [3000][n_mels] (frame-major)."""
    s = power @ fb.T
    lg = np.log10(np.maximum(s, LOG_FLOOR))
    lg = np.maximum(lg, lg.max() - 8.0)
    return (lg + 4.0) / 4.0


def log_mel(pcm: np.ndarray, n_mels: int) -> np.ndarray:
    """One window: pcm (any length, 16 kHz) -> log-mel float32 [3000][n_mels], a frame
    contiguous (the layout [API] gives for wh_encode's input)."""
    x = pad_or_truncate(np.asarray(pcm, dtype=np.float64))
    p = dft_power(frame_signal(x), hann_periodic())
    return log_mel_from_power(p, mel_filterbank(n_mels)).astype(np.float32)


# ========================================================================================
# Encoder  [API] model.nu and kernels.nu; [CKE] "The Encoder", "The Full Stitched Circuit"
# ========================================================================================
def gelu(x: np.ndarray) -> np.ndarray:
    """[API] kernels.nu: GELU with the error function (r11): x * Phi(x)."""
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def layer_norm(x: np.ndarray, g: np.ndarray, b: np.ndarray, eps: float = LN_EPS) -> np.ndarray:
    """[API] kernels.nu: LayerNorm subtracts the mean and has a bias (r10, biased variance)."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * g + b


def conv1d_k3(x: np.ndarray, w: np.ndarray, b: np.ndarray, stride: int) -> np.ndarray:
    """[API] model.nu conv1/conv2: kernel 3, padding 1 (zeros, r9), stride 1 or 2.
    x [T_in][C_in] (time-major), w [C_out][C_in][3] -> [T_out][C_out] with
    y[t][o] = b[o] + sum_{i, j} w[o][i][j] x[stride t + j - 1][i].  Written as an explicit
    im2col (column index i * 3 + j, matching w's flattening) and one matrix product."""
    t_in, c_in = x.shape
    t_out = (t_in + 2 - 3) // stride + 1
    xp = np.zeros((t_in + 2, c_in), dtype=np.float64)
    xp[1:-1] = x
    cols = np.empty((t_out, c_in, 3), dtype=np.float64)
    for j in range(3):
        cols[:, :, j] = xp[j: j + stride * (t_out - 1) + 1: stride]
    return cols.reshape(t_out, c_in * 3) @ w.reshape(w.shape[0], c_in * 3).T.astype(np.float64) + b


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_head: int, return_probs=False):
    """[API] kernels.nu attn_sc / attn_out and [CKE] "The Encoder": NON-causal attention, the
    full T x T square, scores q.k / sqrt(64) (r12), softmax over all keys, times v.
    q, k, v: [T][n_head * 64] -> [T][n_head * 64]."""
    t, d = q.shape
    hd = d // n_head
    out = np.empty((t, d), dtype=np.float64)
    probs = []
    for h in range(n_head):
        sl = slice(h * hd, (h + 1) * hd)
        s = (q[:, sl] @ k[:, sl].T) / np.sqrt(hd)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, sl] = p @ v[:, sl]
        if return_probs:
            probs.append(p)
    return (out, probs) if return_probs else out


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def encoder_block(x: np.ndarray, lw: dict, n_head: int, bk=None) -> np.ndarray:
    """[API] model.nu: x += out_proj(attn(LN1(x))); x += fc2(GELU(fc1(LN2(x)))).
    q, v and out_proj have biases; k_proj has none (bk only exists so a test can show that
    a k bias cannot change the result)."""
    h = layer_norm(x, _f64(lw["ln1_g"]), _f64(lw["ln1_b"]))
    q = h @ _f64(lw["wq"]).T + _f64(lw["bq"])
    k = h @ _f64(lw["wk"]).T
    if bk is not None:
        k = k + _f64(bk)
    v = h @ _f64(lw["wv"]).T + _f64(lw["bv"])
    a = attention(q, k, v, n_head)
    x = x + a @ _f64(lw["wo"]).T + _f64(lw["bo"])
    h = layer_norm(x, _f64(lw["ln2_g"]), _f64(lw["ln2_b"]))
    h = gelu(h @ _f64(lw["w1"]).T + _f64(lw["b1"]))
    return x + h @ _f64(lw["w2"]).T + _f64(lw["b2"])


def encoder_stem(mel: np.ndarray, w: dict) -> np.ndarray:
    """[API] model.nu, [CKE] kernel 7-8: GELU(conv1) -> GELU(conv2, stride 2) -> + stored
    positions (r13).  mel [3000][n_mels] -> x [1500][d]."""
    c1 = gelu(conv1d_k3(_f64(mel), _f64(w["conv1_w"]), _f64(w["conv1_b"]), 1))
    c2 = gelu(conv1d_k3(c1, _f64(w["conv2_w"]), _f64(w["conv2_b"]), 2))
    return c2 + _f64(w["pos"])[: c2.shape[0]]


def encoder(mel: np.ndarray, w: dict, n_head: int) -> np.ndarray:
    """The whole encoder for one window: stem, N blocks, final LayerNorm.
    Returns float64 [1500][d] (the memory the decoder attends to)."""
    x = encoder_stem(mel, w)
    for lw in w["layers"]:
        x = encoder_block(x, lw, n_head)
    return layer_norm(x, _f64(w["lnf_g"]), _f64(w["lnf_b"]))


def encode_window(pcm: np.ndarray, w: dict, n_mels: int, n_head: int):
    """Front end + encoder for one window: returns (log-mel float32, encoder output float64)."""
    mel = log_mel(pcm, n_mels)
    return mel, encoder(mel, w, n_head)


# ========================================================================================
# Shorter encoder context  [README] "Serving" (drafts, whisper.cpp's audio_ctx)
# ========================================================================================
def encoder_ctx(mel: np.ndarray, w: dict, n_head: int, n_ctx: int) -> np.ndarray:
    """The encoder over the first 2 n_ctx log-mel frames of a window (the draft encoder runs
    over the audio heard so far plus 5 s instead of the whole 30 s).  Reading taken: the
    encoder sees only that span, so the convolutions zero-pad at its end exactly as they
    zero-pad at the end of a full window, and the first n_ctx stored positions are added.
    mel [3000][n_mels] -> float64 [n_ctx][d]."""
    return encoder(np.asarray(mel)[: 2 * n_ctx], w, n_head)


# ========================================================================================
# Cross-attention keys and values  [API] model.nu, wh_prepare_cross
# ========================================================================================
def cross_kv(mem: np.ndarray, wk: np.ndarray, wv: np.ndarray, bv=None):
    """One decoder layer's cross-attention keys and values, computed from the encoder memory
    through that layer's own k and v projections ([API] model.nu lists x_wk without a bias,
    x_wv with x_bv).  mem [T][d], wk / wv [d][d] (nn.Linear [out][in]) -> (K, V) [T][d]."""
    m = _f64(mem)
    k = m @ _f64(wk).T
    v = m @ _f64(wv).T
    if bv is not None:
        v = v + _f64(bv)
    return k, v


# ========================================================================================
# One-query attention of a decoder step  [README] "Performance and memory"; [API] wh_decode_step
# ========================================================================================
def attend_one(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_head: int) -> np.ndarray:
    """A single query per head against all the given keys, no mask (the one query sits at the
    end of the sequence): q [n_head * 64], k / v [n_keys][n_head * 64] -> [n_head * 64].
    With no keys the result is zeros (the softmax of an empty set is undefined)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    hd = q.shape[0] // n_head
    out = np.zeros(q.shape[0], dtype=np.float64)
    if k.shape[0] == 0:
        return out
    for h in range(n_head):
        sl = slice(h * hd, (h + 1) * hd)
        s = k[:, sl] @ q[sl] / np.sqrt(hd)
        p = np.exp(s - s.max())
        out[sl] = (p / p.sum()) @ v[:, sl]
    return out


# ========================================================================================
# Upstream front end: 30-s windows of a long clip  [API] main.nu (wh_run); resampling to
# 16 kHz with a windowed sinc  [README] "Transcribing", "How it is verified"
# ========================================================================================
def long_clip_windows(pcm: np.ndarray) -> list:
    """A clip longer than 30 s is cut into consecutive 30-s windows ([API] main.nu, wh_run),
    the last one zero-padded; each window is then an independent 480000-sample input."""
    x = np.asarray(pcm, dtype=np.float32)
    n_win = -(-x.shape[0] // N_SAMPLES)
    out = []
    for w in range(n_win):
        seg = x[w * N_SAMPLES:(w + 1) * N_SAMPLES]
        out.append(np.concatenate([seg, np.zeros(N_SAMPLES - seg.shape[0], np.float32)]))
    return out


def resample_to_16k(x: np.ndarray, rate_in: int) -> np.ndarray:
    """Windowed-sinc resampling to 16 kHz (reading r21: resample_poly's default design, the
    routine the pages check against).  With up / down = 16000 / rate_in in lowest terms and
    M = max(up, down): a low-pass at 1/M of the upsampled Nyquist rate, f sinc(f (t - H)) with
    f = 1/M, H = 10 M, t = 0 .. 2H, times a Kaiser window (beta 5), scaled to unit DC gain and
    then by up.  The output is the zero-phase filtered, upsampled-by-up signal kept every
    down-th sample:  y[j] = sum_i h[j down + H - i up] x[i],  j < ceil(n up / down)."""
    from math import gcd
    x = _f64(x)
    g = gcd(16000, int(rate_in))
    up, down = 16000 // g, int(rate_in) // g
    m_rate = max(up, down)
    half = 10 * m_rate
    t = np.arange(2 * half + 1, dtype=np.float64)
    f = 1.0 / m_rate
    beta = 5.0
    win = np.i0(beta * np.sqrt(np.clip(1.0 - ((t - half) / half) ** 2, 0.0, None))) / np.i0(beta)
    lp = f * np.sinc(f * (t - half))
    h = up * (win * lp) / np.sum(win * lp)
    n = x.shape[0]
    n_out = -(-n * up // down)
    j = np.arange(n_out, dtype=np.int64)
    m = j * down + half
    y = np.zeros(n_out, dtype=np.float64)
    # the sum over i, enumerated by the taps t = m - i up that fall inside the filter
    i_hi = m // up
    for k in range(-(-(2 * half + 1) // up) + 1):
        i = i_hi - k
        tap = m - i * up
        ok = (i >= 0) & (i < n) & (tap <= 2 * half)
        y[ok] += h[tap[ok]] * x[i[ok]]
    return y


# ========================================================================================
# One decoder step  [API] model.nu (decoder weights and state, wh_decode_step, wk_addv_row,
# setrow, wh_argmax); [CKE] "The Full Stitched Circuit" (decoder block: causal self-attention,
# cross-attention into the memory, feed-forward, each with its own LayerNorm and residual;
# final norm and tied output projection), "The Decoder: Write One Token At A Time" and
# "Decoding Token By Token" (the self-attention cache grows by one row per step)
# ========================================================================================
def decoder_embed(tok: int, pos: int, w: dict) -> np.ndarray:
    """The token's row of the embedding plus row `pos` of the decoder's stored positions
    ([API] wk_addv_row: x += embed_positions[pos])."""
    return _f64(w["tok_embd"])[tok] + _f64(w["dec_pos"])[pos]


def decoder_self_attention(h: np.ndarray, lw: dict, kcache: np.ndarray, vcache: np.ndarray, pos: int,
                           n_head: int) -> np.ndarray:
    """Self-attention of the token at position `pos` (reading r23).  Its own key and value
    (k has no bias, like the encoder's) are written into row `pos` of the layer's caches
    ([API] setrow), then its query attends over rows 0..pos -- what came before it plus
    itself.  One query at the end needs no mask ([API] wh_decode_step); rows past `pos` are
    never read.  kcache / vcache [n_text_ctx][d] are modified in place."""
    q = h @ _f64(lw["wq"]).T + _f64(lw["bq"])
    kcache[pos] = h @ _f64(lw["wk"]).T
    vcache[pos] = h @ _f64(lw["wv"]).T + _f64(lw["bv"])
    return attend_one(q, kcache[: pos + 1], vcache[: pos + 1], n_head)


def decoder_block_step(x: np.ndarray, lw: dict, kcache, vcache, pos: int, xk, xv, n_head: int) -> np.ndarray:
    """One decoder block for one token ([CKE] "The Full Stitched Circuit"):
    x += out(self-attn(LN1 x)); x += x_out(cross-attn(LNx x) over the memory's cached K/V);
    x += fc2(GELU(fc1(LN2 x))).  The cross query has a bias, its keys none ([API] model.nu)."""
    h = layer_norm(x, _f64(lw["ln1_g"]), _f64(lw["ln1_b"]))
    a = decoder_self_attention(h, lw, kcache, vcache, pos, n_head)
    x = x + a @ _f64(lw["wo"]).T + _f64(lw["bo"])
    h = layer_norm(x, _f64(lw["lnx_g"]), _f64(lw["lnx_b"]))
    q = h @ _f64(lw["xwq"]).T + _f64(lw["xbq"])
    a = attend_one(q, xk, xv, n_head)
    x = x + a @ _f64(lw["xwo"]).T + _f64(lw["xbo"])
    h = layer_norm(x, _f64(lw["ln2_g"]), _f64(lw["ln2_b"]))
    return x + gelu(h @ _f64(lw["w1"]).T + _f64(lw["b1"])) @ _f64(lw["w2"]).T + _f64(lw["b2"])


def decode_step(tok: int, pos: int, w: dict, kcache: list, vcache: list, xk: list, xv: list,
                n_head: int) -> np.ndarray:
    """[API] wh_decode_step for one sequence: token `tok` at position `pos`, with positions
    0..pos-1 already in the self-attention caches.  Runs every decoder block (appending this
    token's keys and values to kcache[l] / vcache[l], each [n_text_ctx][d], in place), the
    final LayerNorm and the output projection through the token embedding (Whisper ties
    them).  xk[l] / xv[l] [n_ctx][d] are decoder layer l's cross-attention keys and values
    (cross_kv of the encoder memory).  Returns the logits, float64 [n_vocab]."""
    x = decoder_embed(tok, pos, w)
    for l, lw in enumerate(w["layers"]):
        x = decoder_block_step(x, lw, kcache[l], vcache[l], pos, xk[l], xv[l], n_head)
    x = layer_norm(x, _f64(w["lnf_g"]), _f64(w["lnf_b"]))
    return _f64(w["tok_embd"]) @ x


def greedy_token(logits: np.ndarray) -> int:
    """[API] wh_argmax: the index of the largest logit (the first one on a tie)."""
    return int(np.argmax(logits))
