/*
 * wh.h -- C ABI of libwh.so: the Whisper audio-encoder forward pass on one GB300 (sm_103a).
 *
 * The path: 16 kHz PCM -> log-mel (wh_frontend) -> conv stem + N pre-LN encoder blocks +
 * final LayerNorm (wh_encode) -> the 1500 x d_model memory the decoder attends to.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers unless stated otherwise.  The caller owns every
 *     buffer (inputs, outputs, weights, workspace); the library never frees or keeps them.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*, NULL = the legacy
 *     default stream).  Argument errors are detected on the host and returned before anything
 *     is launched.  Errors found on the device (a bounded wait that ran out, a bounds check)
 *     are recorded in a per-device status word and returned by wh_status().
 *   - The library's own persistent state is small constant tables (Hann window, twiddles,
 *     mel filterbanks) in static device arrays, set up on the first call on each device.
 *     Make that first call outside any CUDA-graph capture.
 *   - Matrices are bfloat16 (passed as wh_bf16 bit patterns), vectors are float32,
 *     accumulation is float32, the residual stream is float32.
 *   - Return value: WH_OK (0) or one of the WH_E* codes below; wh_strerror() names them.
 */
#ifndef WH_H
#define WH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    WH_OK = 0,
    WH_EINVAL = 1,     /* bad argument: null pointer, unsupported shape, misaligned buffer */
    WH_ENOSPC = 2,     /* workspace smaller than the matching *_workspace() size */
    WH_ECUDA = 3,      /* a CUDA runtime call or launch failed */
    WH_ETIMEOUT = 4,   /* a device-side bounded wait ran out (reported by wh_status) */
    WH_EBOUNDS = 5,    /* a device-side bounds check fired (reported by wh_status) */
    WH_ENODEV = 6      /* no usable CUDA device */
};

typedef uint16_t wh_bf16;   /* bfloat16 bit pattern */

/* Encoder hyper-parameters ("whisper 0.9.0 API", model.nu: the shape is read from the
 * checkpoint, not hard-coded).  head_dim = d_model / n_head must be 64; n_mels is 80 or 128
 * ("How Audio Becomes Words", section "Tiny, Base, Small, Large": large-v3 uses 128 bins);
 * d_model and d_ff multiples of 128, d_model <= 2048.  n_layer may be 0 (stem + final norm).
 * The encoder context is fixed at 1500 positions. */
typedef struct {
    int n_mels, d_model, n_head, n_layer, d_ff;
} wh_config;

/* One encoder block ("whisper 0.9.0 API", model.nu: N x [LN -> self-attn -> +residual,
 * LN -> fc1 -> GELU -> fc2 -> +residual]).  Matrices use the nn.Linear layout [out][in],
 * row-major.  q, v and out_proj have a bias; the key projection has none (model.nu lists
 * no k bias among the weights), so there is no bk field. */
typedef struct {
    const float *ln1_g, *ln1_b;            /* [d] */
    const wh_bf16 *wq, *wk, *wv;           /* [d][d] each */
    const float *bq, *bv;                  /* [d] */
    const wh_bf16 *wo;  const float *bo;   /* [d][d], [d] */
    const float *ln2_g, *ln2_b;            /* [d] */
    const wh_bf16 *w1;  const float *b1;   /* fc1: [d_ff][d], [d_ff] */
    const wh_bf16 *w2;  const float *b2;   /* fc2: [d][d_ff], [d] */
} wh_layer_weights;

/* All encoder weights.  `layers` is a HOST array of n_layer structs (of device pointers).
 * Conv weights use the PyTorch Conv1d layout [c_out][c_in][3] (the pages give no layout). */
typedef struct {
    const wh_bf16 *conv1_w; const float *conv1_b;   /* [d][n_mels][3], [d] */
    const wh_bf16 *conv2_w; const float *conv2_b;   /* [d][d][3], [d] */
    const float *pos;                               /* stored positions [1500][d] */
    const wh_layer_weights *layers;                 /* host array [n_layer] */
    const float *lnf_g, *lnf_b;                     /* final LayerNorm [d] */
} wh_weights;

/* ---------------------------------------------------------------------------------------
 * Front end.  "How Audio Becomes Words", section "The Frontend: Sound Becomes A Tensor",
 * kernels 3-6: pad or truncate to 480000 samples; reflect padding, periodic Hann(400),
 * n_fft 400, hop 160 -> a 201 x 3000 power grid; Slaney mel filters (area-normalised) to
 * n_mels bins; log10, a clamp at (window maximum - 8) (-80 dB, relative to the loudest
 * point of the whole clip) and (x + 4) / 4.
 *
 *   pcm   device float32 [batch][n]: window b's samples start at pcm + b * n.  n >= 0;
 *         n < 480000 reads zeros past the end, n > 480000 ignores the rest.
 *   mel   device float32 [batch][3000][n_mels]: per window 3000 rows of n_mels values, each
 *         frame contiguous (the layout "whisper 0.9.0 API" gives for wh_encode's input).
 *   workspace  device scratch of at least wh_frontend_workspace(batch) bytes, 16-byte aligned
 *         (the per-window maxima and the kernel's grid-barrier count: batch + 1 words);
 *         contents need not be initialised.
 * The work is one cooperative launch (every block resident at once) with a grid-wide barrier
 * between the log10 values and the clamp; the barrier's wait is bounded (1 s): if it runs
 * out, wh_status() reports WH_ETIMEOUT and the output is left unclamped.
 * Errors: WH_EINVAL (null pointer with batch > 0, n < 0, batch < 0 or > 65535, n_mels not
 *         80/128), WH_ENOSPC (workspace too small), WH_ECUDA.  batch == 0 is a no-op.
 * ------------------------------------------------------------------------------------ */
size_t wh_frontend_workspace(int batch);
int wh_frontend(const float *pcm, int64_t n, int batch, int n_mels, float *mel,
                void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * Front end of one long clip ("whisper 0.9.0 API", main.nu, wh_run: audio longer than 30 s is
 * cut into 30-s windows, each encoded -- and decoded -- on its own).  Window w holds samples
 * [480000 w, 480000 (w + 1)) of the clip, the last one zero-padded; each window gets its own
 * log-mel exactly as wh_frontend computes it (own reflect padding, own maximum and clamp).
 *   wh_frontend_windows(n_total) = ceil(n_total / 480000) (0 for an empty clip).
 *   pcm   device float32 [n_total], 16-byte aligned
 *   mel   device float32 [wh_frontend_windows(n_total)][3000][n_mels]
 *   workspace >= wh_frontend_workspace(windows) bytes, 16-byte aligned.
 * Errors: WH_EINVAL (null or misaligned pointer, n_total < 0, more than 65535 windows, n_mels
 * not 80/128), WH_ENOSPC, WH_ECUDA.  An empty clip is a no-op.
 * ------------------------------------------------------------------------------------ */
int64_t wh_frontend_windows(int64_t n_total);
int wh_frontend_long(const float *pcm, int64_t n_total, int n_mels, float *mel, void *workspace,
                     size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * Resampling to 16 kHz ("whisper" package page, "Transcribing": input at any rate is
 * resampled to 16 kHz with a windowed sinc, not linear interpolation; "How it is verified":
 * checked against scipy's resample_poly).  The filter is resample_poly's default design: with
 * up / down = 16000 / rate_in in lowest terms and M = max(up, down), a Kaiser-windowed
 * (beta 5) sinc low-pass at 1 / M of the upsampled Nyquist rate, 20 M + 1 taps, unit DC gain,
 * times up; y[j] = sum_i h[j down + 10 M - i up] x[i] (zero phase, x = 0 outside the clip).
 *   wh_resample_length(n_in, rate_in) = ceil(n_in * up / down) output samples (-1 for bad
 *   arguments); wh_resample_workspace(rate_in) bytes of workspace hold the polyphase table
 *   (built on the device by every call; 16-byte aligned).
 *   x     device float32 [batch][n_in] at rate_in Hz, 1000 <= rate_in <= 384000
 *   y     device float32 [batch][wh_resample_length(n_in, rate_in)] at 16 kHz
 * Errors: WH_EINVAL, WH_ENOSPC, WH_ECUDA.  batch == 0 or n_in == 0 is a no-op.
 * ------------------------------------------------------------------------------------ */
int64_t wh_resample_length(int64_t n_in, int rate_in);
size_t wh_resample_workspace(int rate_in);
int wh_resample(const float *x, int64_t n_in, int batch, int rate_in, float *y, void *workspace,
                size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * wh_frontend_static: wh_frontend for callers that cannot allocate device memory.
 * (The pages have no counterpart: this is an interface choice of this library.)
 * Some callers cannot hand the library a scratch buffer at the point they call in: a
 * real-time audio callback must not block on the CUDA allocator, and a process that gave
 * all of its device memory to another allocator up front has none left.  This variant keeps
 * the per-window maxima in a fixed array inside the library (WH_FRONTEND_STATIC_MAX_BATCH + 1
 * words, held on every GPU that loads the library until the process exits) and allocates
 * nothing; pcm and mel are as for wh_frontend.
 *   - batch > WH_FRONTEND_STATIC_MAX_BATCH returns WH_ENOSPC (nothing is launched).
 *   - The first call on each device sets up the library's tables and looks up the array's
 *     device address; make that first call before any stream capture.
 *   - All calls on a device share the array: calls that overlap on the GPU (for example on
 *     two streams at once) race on it.  Each call clears the maxima before using them.
 * Errors: as wh_frontend, plus WH_ENOSPC for an oversized batch.
 * ------------------------------------------------------------------------------------ */
#define WH_FRONTEND_STATIC_MAX_BATCH 4096
int wh_frontend_static(const float *pcm, int64_t n, int batch, int n_mels, float *mel, void *stream);

/* ---------------------------------------------------------------------------------------
 * Encoder.  "whisper 0.9.0 API", model.nu: conv1 (k=3, s=1, pad=1) n_mels -> d, GELU;
 * conv2 (k=3, s=2, pad=1) d -> d, GELU, 3000 -> 1500 frames; + stored positions; n_layer
 * pre-LN blocks with NON-causal self-attention (scores q.k / sqrt(64), kernels.nu); final
 * LayerNorm (eps 1e-5); GELU is the erf form (kernels.nu).
 *
 *   mel   device float32 [batch][3000][n_mels] (as produced by wh_frontend)
 *   out   device float32 [batch][1500][d_model], row-major (the encoder-state layout of
 *         "whisper 0.9.0 API", wh_enc_out); may not alias mel or the workspace.
 *   workspace  device scratch of at least wh_encode_workspace(cfg, batch) bytes, 256-byte
 *         aligned; contents need not be initialised; not to be shared by concurrent calls.
 * Errors: WH_EINVAL (null pointer, unsupported config, misaligned pointer), WH_ENOSPC,
 *         WH_ECUDA.  batch == 0 is a no-op.
 * ------------------------------------------------------------------------------------ */
size_t wh_encode_workspace(const wh_config *cfg, int batch);
int wh_encode(const float *mel, int batch, const wh_config *cfg, const wh_weights *w,
              float *out, void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * Encoder over a shorter context (the "whisper" package page, "Serving": drafts run the
 * encoder over the audio heard so far plus 5 s, at least 10 s, instead of the full 30 s --
 * whisper.cpp's audio_ctx).  The encoder reads only the first 2 n_ctx log-mel frames of each
 * window, pads that span with zeros at both ends for the convolutions (as it pads the full
 * window), adds the first n_ctx stored positions and attends over n_ctx positions.
 * n_ctx = 1500 is wh_encode exactly.
 *   mel   device float32 [batch][3000][n_mels], as for wh_encode (windows 3000 frames apart;
 *         frames 2 n_ctx .. 2999 are not read)
 *   out   device float32 [batch][n_ctx][d_model], row-major
 *   1 <= n_ctx <= 1500; workspace >= wh_encode_ctx_workspace(cfg, batch, n_ctx) bytes,
 *   256-byte aligned.  Errors as wh_encode, WH_EINVAL for n_ctx out of range.
 * ------------------------------------------------------------------------------------ */
size_t wh_encode_ctx_workspace(const wh_config *cfg, int batch, int n_ctx);
int wh_encode_ctx(const float *mel, int batch, int n_ctx, const wh_config *cfg, const wh_weights *w,
                  float *out, void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * Cross-attention keys and values of every decoder layer ("whisper 0.9.0 API", model.nu,
 * wh_prepare_cross: the decoder's cross-attention reads the encoder memory through its own
 * k and v projections, and since the memory does not change while a clip is transcribed they
 * are computed once per clip rather than once per generated token).  For decoder layer l:
 *   K_l = mem Wk_l^T           (the cross k projection has no bias, model.nu)
 *   V_l = mem Wv_l^T + bv_l
 *   mem   device float32 [batch * n_ctx][d_model] (wh_encode's or wh_encode_ctx's output);
 *         rounded once to bf16 as the tensor-core operand
 *   w     host struct of host arrays of n_layer DEVICE pointers: wk[l], wv[l] bf16 [d][d]
 *         (nn.Linear [out][in]), bv[l] float32 [d] or NULL (no bias)
 *   kv    device bf16 [n_layer][batch * n_ctx][2 d_model]: row r of layer l holds K_l[r] in
 *         columns 0 .. d-1 and V_l[r] in columns d .. 2d-1 (head h: 64 h .. 64 h + 63 of each)
 *   workspace  >= wh_prepare_cross_workspace(batch, n_ctx, d_model) bytes, 256-byte aligned
 *   d_model a multiple of 128 in [128, 2048]; 1 <= n_ctx <= 1500; n_layer >= 0.
 * Errors: WH_EINVAL (null or misaligned pointer, shape out of range), WH_ENOSPC, WH_ECUDA.
 * batch == 0 or n_layer == 0 is a no-op.
 * ------------------------------------------------------------------------------------ */
typedef struct {
    const wh_bf16 *const *wk;   /* host array [n_layer] of device [d][d] */
    const wh_bf16 *const *wv;   /* host array [n_layer] of device [d][d] */
    const float *const *bv;     /* host array [n_layer] of device [d] (entries may be NULL) */
} wh_cross_weights;
size_t wh_prepare_cross_workspace(int batch, int n_ctx, int d_model);
int wh_prepare_cross(const float *mem, int batch, int n_ctx, int d_model, int n_layer,
                     const wh_cross_weights *w, wh_bf16 *kv, void *workspace, size_t ws_bytes,
                     void *stream);

/* ---------------------------------------------------------------------------------------
 * Recorded passes (the "whisper" package page, "Implementation notes", records its encoder
 * pass once when a model is opened and replays it per request).  wh_graph_capture records one
 * wh_frontend + wh_encode pass on `stream` into a CUDA graph (arguments exactly as for those
 * two calls; mel is the log-mel buffer between them).  wh_graph_launch replays it on any
 * stream: the same buffers are read and written, so refresh pcm in place and replay.  The
 * graph keeps the pointers it was recorded with; buffers must stay alive until
 * wh_graph_destroy.  `stream` must not be the legacy default stream (NULL).
 * Errors: as wh_frontend / wh_encode; WH_EINVAL for a NULL stream or graph; WH_ECUDA if the
 * capture or instantiation fails.
 * ------------------------------------------------------------------------------------ */
typedef struct wh_graph wh_graph;
int wh_graph_capture(const float *pcm, int64_t n, int batch, const wh_config *cfg, const wh_weights *w,
                     float *mel, float *out, void *fe_ws, size_t fe_ws_bytes, void *enc_ws, size_t enc_ws_bytes,
                     void *stream, wh_graph **graph);
/* The encoder alone (wh_encode's arguments): mel is the recorded pass's input. */
int wh_graph_capture_encode(const float *mel, int batch, const wh_config *cfg, const wh_weights *w,
                            float *out, void *enc_ws, size_t enc_ws_bytes, void *stream, wh_graph **graph);
int wh_graph_launch(wh_graph *graph, void *stream);
int wh_graph_destroy(wh_graph *graph);

/* ---------------------------------------------------------------------------------------
 * Single steps of the encoder, exposed for testing and for callers that compose their own
 * pipeline.  Same conventions as above.
 * ------------------------------------------------------------------------------------ */

/* LayerNorm ("whisper 0.9.0 API", kernels.nu: it subtracts the mean and has a bias):
 * y[r] = (x[r] - mean) / sqrt(var + 1e-5) * g + b over d columns, biased variance.
 * x float32 [rows][d]; y is bf16 (y_bf16 = 1) or float32 (y_bf16 = 0) [rows][d].
 * d a multiple of 64, 64 <= d <= 2048. */
int wh_layer_norm(const float *x, int rows, int d, const float *g, const float *b,
                  void *y, int y_bf16, void *stream);

/* Dense layer on the tensor cores: acc[r][c] = sum_k a[r][k] * w[c][k] (nn.Linear [out][in]).
 * a bf16 [rows][k], w bf16 [n][k]; k a multiple of 8, n a multiple of 128.
 *   WH_EPI_BF16        y bf16 [rows][n] = acc + bias
 *   WH_EPI_GELU_BF16   y bf16 [rows][n] = GELU(acc + bias)      (fc1)
 *   WH_EPI_RESID_F32   y float32 [rows][n] += acc + bias       (out_proj, fc2)
 * bias may be NULL (no bias). */
enum { WH_EPI_BF16 = 0, WH_EPI_GELU_BF16 = 1, WH_EPI_RESID_F32 = 2 };
int wh_linear(const wh_bf16 *a, int rows, int k, const wh_bf16 *w, int n, const float *bias,
              int epilogue, void *y, void *stream);

/* Non-causal multi-head attention over all n_ctx keys ("whisper 0.9.0 API", kernels.nu,
 * attn_f / attn_sc / attn_out with causal = 0): for each window b and head h,
 * o = softmax(q k^T / sqrt(64)) v.  qkv bf16 [batch * n_ctx][3 * n_head * 64] with the q,
 * k and v of head h in columns 64 h, D + 64 h and 2 D + 64 h (D = 64 n_head);
 * out bf16 [batch * n_ctx][D].  1 <= n_ctx <= 1500. */
int wh_attention(const wh_bf16 *qkv, int batch, int n_ctx, int n_head, wh_bf16 *out,
                 void *stream);

/* One-query attention of a decoder step ("whisper" package page, "Performance and memory":
 * a decode step has one query per head, so the keys are split across blocks and the blocks'
 * partial softmaxes are merged; "whisper 0.9.0 API", wh_decode_step: with the single query at
 * the end, the decoder's self-attention needs no mask, and its cross-attention reads every
 * encoder position).  For each sequence b and head h:
 *   out[b][64 h ..] = softmax(q[b][64 h ..] . K_b,h^T / sqrt(64)) V_b,h    over n_keys[b] keys
 *   q     device bf16 [batch][64 n_head]
 *   k, v  device bf16: key t of sequence b, head h is the 64 values at
 *         k + b * seq_stride + t * row_stride + 64 h (likewise v).  wh_prepare_cross's rows
 *         give row_stride = 2 d_model, seq_stride = n_ctx * 2 d_model, v = k + d_model; a
 *         self-attention cache [batch][max][d_model] gives row_stride = d_model.
 *   n_keys  device int32 [batch], or NULL: max_keys for all.  A sequence with no keys gets
 *         zeros.  The counts live in device memory, so they are checked on the device: a
 *         count below 0 or above max_keys is clamped to that range (nothing outside it is
 *         read) and recorded as WH_EBOUNDS, which wh_status() then returns.
 *   out   device bf16 [batch][64 n_head]
 *   workspace  >= wh_decode_attention_workspace(batch, n_head, max_keys) bytes, 256-byte
 *         aligned, contents need not be initialised; not shared by concurrent calls.
 *   row_stride >= 64 n_head and seq_stride >= 0, both multiples of 8 elements; pointers
 *   16-byte aligned; 1 <= max_keys <= 2^30; batch, n_head <= 65535.
 * Errors: WH_EINVAL, WH_ENOSPC, WH_ECUDA.  batch == 0 is a no-op. */
size_t wh_decode_attention_workspace(int batch, int n_head, int max_keys);
int wh_decode_attention(const wh_bf16 *q, const wh_bf16 *k, const wh_bf16 *v, int64_t row_stride,
                        int64_t seq_stride, const int *n_keys, int max_keys, int batch, int n_head,
                        wh_bf16 *out, void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * One decoder step for a batch of sequences ("whisper 0.9.0 API", model.nu, wh_decode_step:
 * token tok at position pos, everything before it already in the KV cache, the logits left
 * on the device; wk_addv_row adds the stored position row; setrow writes the token's key and
 * value into the cache; wh_argmax is greedy decoding.  "How Audio Becomes Words", "The Full
 * Stitched Circuit": a decoder block is causal self-attention, cross-attention into the
 * encoder memory and a feed-forward, each behind its own LayerNorm and added to the residual;
 * then a final LayerNorm and the output projection through the token embedding).
 *
 * For each sequence b, with t = tok[b] and p = pos[b]:
 *   x = tok_embd[t] + pos_embd[p]
 *   per layer l:  h = LN1(x); q = h Wq^T + bq; k = h Wk^T (no bias); v = h Wv^T + bv;
 *                 kcache[l][b][p] = k, vcache[l][b][p] = v;
 *                 x += attend(q, kcache[l][b][0..p], vcache[l][b][0..p]) Wo^T + bo
 *                 h = LNx(x); x += attend(h Wxq^T + bxq, cross K_l, V_l of window b) Wxo^T + bxo
 *                 h = LN2(x); x += GELU(h W1^T + b1) W2^T + b2
 *   logits[b] = LNf(x) tok_embd^T;  next_tok[b] = the index of the first largest logit
 * attend(q, K, V) is per head h: softmax(q_h K_h^T / sqrt(64)) V_h.  Rows of the self-attention
 * caches past p are never read.  Tokens, positions, caches and logits stay on the device, so a
 * decode loop needs no host round trip: the caller writes next_tok into tok and pos + 1 into
 * pos (or records the step once in a CUDA graph and replays it).
 *
 *   tok, pos   device int32 [batch]: a token outside 0 .. n_vocab-1 or a position outside
 *              0 .. n_text_ctx-1 is clamped into range (nothing outside a table or cache is
 *              touched) and recorded as WH_EBOUNDS, which wh_status() then returns.
 *   kcache, vcache  device bf16 [n_layer][batch][n_text_ctx][d_model]; row pos[b] of every
 *              layer is written, rows 0 .. pos[b]-1 are read.
 *   cross_kv   device bf16 [n_layer][batch * n_ctx][2 d_model]: wh_prepare_cross's output
 *              (K in columns 0 .. d-1, V in d .. 2d-1), sequence b reading window b's rows.
 *   logits     device float32 [batch][n_vocab];  next_tok  device int32 [batch] or NULL.
 *   workspace  >= wh_decode_step_workspace(cfg, batch) bytes, 256-byte aligned, contents
 *              need not be initialised; not shared by concurrent calls.
 *   d_model a multiple of 128 in [128, 2048] with head_dim 64; d_ff a multiple of 128;
 *   1 <= batch <= 256; 1 <= n_ctx <= 1500.  Matrices bf16 [out][in], vectors float32.
 * Precision: bf16 operands on the tensor cores with fp32 accumulation, the residual stream in
 * fp32, LayerNorm outputs, q / k / v, attention outputs and the caches in bf16.
 * Errors: WH_EINVAL (null or misaligned pointer, shape out of range), WH_ENOSPC, WH_ECUDA.
 * batch == 0 is a no-op.
 * ------------------------------------------------------------------------------------ */
typedef struct {
    int d_model, n_head, n_layer, d_ff, n_vocab, n_text_ctx;
} wh_dec_config;
typedef struct {
    const float *ln1_g, *ln1_b;                  /* self-attention LayerNorm [d] */
    const wh_bf16 *wq, *wk, *wv;                 /* [d][d] each (no k bias) */
    const float *bq, *bv;                        /* [d] */
    const wh_bf16 *wo;  const float *bo;         /* [d][d], [d] */
    const float *lnx_g, *lnx_b;                  /* cross-attention LayerNorm [d] */
    const wh_bf16 *xwq; const float *xbq;        /* cross query [d][d], [d] */
    const wh_bf16 *xwo; const float *xbo;        /* cross output [d][d], [d] */
    const float *ln2_g, *ln2_b;                  /* feed-forward LayerNorm [d] */
    const wh_bf16 *w1;  const float *b1;         /* [d_ff][d], [d_ff] */
    const wh_bf16 *w2;  const float *b2;         /* [d][d_ff], [d] */
} wh_dec_layer_weights;
typedef struct {
    const wh_bf16 *tok_embd;                     /* [n_vocab][d]: embedding and output projection */
    const float *pos;                            /* stored decoder positions [n_text_ctx][d] */
    const wh_dec_layer_weights *layers;          /* HOST array [n_layer] */
    const float *lnf_g, *lnf_b;                  /* final LayerNorm [d] */
} wh_dec_weights;
size_t wh_decode_step_workspace(const wh_dec_config *cfg, int batch);
int wh_decode_step(const int *tok, const int *pos, int batch, const wh_dec_config *cfg, const wh_dec_weights *w,
                   wh_bf16 *kcache, wh_bf16 *vcache, const wh_bf16 *cross_kv, int n_ctx, float *logits,
                   int *next_tok, void *workspace, size_t ws_bytes, void *stream);
/* One decoder step recorded into a CUDA graph (wh_decode_step's arguments; replay with
 * wh_graph_launch, free with wh_graph_destroy; stream not NULL).  tok and pos are read from
 * device memory at every replay, so a decode loop refreshes them in place (next_tok -> tok,
 * pos + 1 -> pos) and replays; the caches, cross K/V, logits and workspace are the recorded
 * buffers. */
int wh_graph_capture_decode(const int *tok, const int *pos, int batch, const wh_dec_config *cfg,
                            const wh_dec_weights *w, wh_bf16 *kcache, wh_bf16 *vcache, const wh_bf16 *cross_kv,
                            int n_ctx, float *logits, int *next_tok, void *workspace, size_t ws_bytes, void *stream,
                            wh_graph **graph);

/* ---------------------------------------------------------------------------------------
 * Status, errors, tracing
 * ------------------------------------------------------------------------------------ */

/* Synchronises `stream`, then returns and clears the current device's status word:
 * WH_OK, WH_ETIMEOUT or WH_EBOUNDS (or WH_ECUDA if the synchronisation failed). */
int wh_status(void *stream);

/* Forgets the library's per-device set-up (kernel attributes, status-word address, the
 * constant tables' "ready" mark) and its host-side caches; the next call on a device sets it
 * up again.  The constant tables are static device arrays: nothing is freed, nothing the
 * caller owns is touched, and no device is reset.  Call it with no call of this library in
 * flight (after a stream synchronisation). */
int wh_shutdown(void);

/* A static, NUL-terminated name for a WH_* code. */
const char *wh_strerror(int code);

/* Self-test of the bounded-wait machinery: launches one block that waits on a barrier that
 * nothing completes, with a wait limit of `limit_ns` nanoseconds (<= 1e9).  The wait runs
 * out, the block records WH_ETIMEOUT in the status word and returns; wh_status() then
 * reports it.  Does not fault or hang the GPU. */
int wh_selftest_timeout(uint64_t limit_ns, void *stream);

/* Per-kernel timing with CUDA events recorded around each launch on the launching stream.
 * wh_trace_enable(1) starts recording (clearing earlier records), 0 stops.  wh_trace_read
 * synchronises the recorded events and fills up to `max` entries (one per kernel class)
 * with launch counts, total device milliseconds and algorithmic work; returns the number of
 * classes, or a negative WH_E* code. */
typedef struct {
    char name[32];        /* kernel class: "gemm", "attention", "layernorm", "frontend", ... */
    int launches;
    double total_ms;
    double flops;         /* algorithmic flops of all recorded launches */
    double bytes;         /* algorithmic HBM bytes of all recorded launches */
} wh_trace_stat;
int wh_trace_enable(int on);
int wh_trace_read(wh_trace_stat *out, int max);

/* Number of kernels the library launched since the last call (all devices, all streams). */
int64_t wh_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* WH_H */
