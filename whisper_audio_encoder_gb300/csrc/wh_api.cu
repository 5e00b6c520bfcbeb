// C ABI of libwh.so (declared in include/wh.h): argument validation, per-device state,
// workspace layout, the encoder's launch sequence, status word and per-kernel tracing.
//
// Launch sequence of wh_encode ("whisper 0.9.0 API", model.nu; "How Audio Becomes Words",
// section "The Full Stitched Circuit"):
//   repack conv weights -> mel im2col -> conv1 GEMM (+GELU, into conv2's im2col)
//   -> conv2 GEMM (+GELU +positions, fp32 residual stream x)
//   -> per block: LN1 -> QKV GEMM (+bq, +bv) -> attention -> out_proj GEMM (+bo, +x)
//                 -> LN2 -> fc1 GEMM (+b1, GELU) -> fc2 GEMM (+b2, +x)
//   -> final LN (fp32 out).
// Everything runs on the caller's stream; nothing allocates device memory.
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace wh {

__device__ int g_status;   // per-device status word

namespace {

constexpr int N_CTX = 1500, N_FRAMES = 3000;
constexpr int MAX_DEV = 64;
constexpr unsigned long long DEFAULT_WAIT_NS = 1000000000ull;  // 1 s per bounded wait

struct DevState {
    bool ready = false;
    int *status = nullptr;
    int num_sms = 0;
};
DevState g_dev[MAX_DEV];
std::mutex g_dev_mu;
std::atomic<long long> g_launches{0};

int ensure_device(DevState **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) {
        cudaGetLastError();
        return WH_ENODEV;
    }
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
        cudaGetLastError();
        return WH_ENODEV;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevState &st = g_dev[dev];
    if (!st.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return WH_ECUDA;
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return WH_ECUDA;
        if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return WH_ECUDA;
        if (int rc = frontend_init_tables()) return rc;
        if (int rc = gemm_prepare(st.num_sms)) return rc;
        if (int rc = attention_prepare()) return rc;
        if (int rc = resample_prepare()) return rc;
        if (int rc = dec_gemm_prepare()) return rc;
        st.status = static_cast<int *>(p);
        st.ready = true;
    }
    *out = &st;
    return WH_OK;
}

DevCtl ctl_of(const DevState *st, unsigned long long wait_ns = DEFAULT_WAIT_NS) {
    DevCtl c;
    c.status = st->status;
    c.wait_ns = wait_ns;
    return c;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

// ---- tracing ---------------------------------------------------------------------------
struct TraceRec {
    int cls;
    cudaEvent_t e0, e1;
    double flops, bytes;
};
const char *const kTraceNames[TR_NCLASS] = {"frontend", "stem_prep", "gemm",       "attention",
                                             "layernorm", "gemm_conv", "gemm_qkv",   "gemm_out",
                                             "gemm_fc1",  "gemm_fc2",  "cross_prep", "gemm_cross",
                                             "decode_attention", "resample", "dec_gemm", "dec_other"};
std::mutex g_tr_mu;
bool g_tr_on = false;
std::vector<TraceRec> g_tr;
std::vector<cudaEvent_t> g_tr_pool;
size_t g_tr_used = 0;
cudaEvent_t g_tr_open = nullptr;
constexpr size_t TRACE_MAX_EVENTS = 16384;

cudaEvent_t tr_event() {
    if (g_tr_used < g_tr_pool.size()) return g_tr_pool[g_tr_used++];
    if (g_tr_pool.size() >= TRACE_MAX_EVENTS) return nullptr;
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_tr_pool.push_back(e);
    ++g_tr_used;
    return e;
}

// ---- config validation -----------------------------------------------------------------
int check_config(const wh_config *c) {
    if (!c) return WH_EINVAL;
    if (c->n_mels != 80 && c->n_mels != 128) return WH_EINVAL;
    if (c->d_model <= 0 || c->d_model % 128 != 0 || c->d_model > 2048) return WH_EINVAL;
    if (c->n_head <= 0 || c->d_model != 64 * c->n_head) return WH_EINVAL;
    if (c->n_layer < 0 || c->d_ff <= 0 || c->d_ff % 128 != 0) return WH_EINVAL;
    return WH_OK;
}

struct EncLayout {
    size_t x, xn, qkv, ao, h, a1, w1p, w2p, sk, skt, total;
};

// n_ctx encoder positions per window (conv1 runs over 2 n_ctx log-mel frames)
EncLayout layout(const wh_config *c, int batch, int n_ctx) {
    const size_t rows = (size_t)batch * n_ctx, d = c->d_model, f = c->d_ff, M = c->n_mels;
    EncLayout L;
    size_t off = 0;
    L.x = off;   off += up256(rows * d * 4);
    L.xn = off;  off += up256(rows * d * 2);
    L.qkv = off; off += up256(rows * 3 * d * 2);   // also conv2's im2col matrix
    L.ao = off;  off += up256(rows * d * 2);
    L.h = off;   off += up256(rows * f * 2);
    L.a1 = off;  off += up256((size_t)batch * 2 * n_ctx * 3 * M * 2);
    L.w1p = off; off += up256(d * 3 * M * 2);
    L.w2p = off; off += up256(d * 3 * d * 2);
    L.sk = off;  off += up256(gemm_sk_bytes((long long)rows, (int)d));   // stream-K partials of out_proj / fc2
    L.skt = off; off += up256(gemm_sk_ticket_bytes((long long)rows, (int)d));
    L.total = off;
    return L;
}

bool vec_ok(const float *p) { return p != nullptr && aligned(p, 16); }
bool mat_ok(const wh_bf16 *p) { return p != nullptr && aligned(p, 16); }

int check_weights(const wh_config *c, const wh_weights *w) {
    if (!w) return WH_EINVAL;
    if (!mat_ok(w->conv1_w) || !vec_ok(w->conv1_b) || !mat_ok(w->conv2_w) || !vec_ok(w->conv2_b) ||
        !vec_ok(w->pos) || !vec_ok(w->lnf_g) || !vec_ok(w->lnf_b))
        return WH_EINVAL;
    if (c->n_layer > 0 && !w->layers) return WH_EINVAL;
    for (int l = 0; l < c->n_layer; ++l) {
        const wh_layer_weights &L = w->layers[l];
        if (!vec_ok(L.ln1_g) || !vec_ok(L.ln1_b) || !mat_ok(L.wq) || !mat_ok(L.wk) || !mat_ok(L.wv) ||
            !vec_ok(L.bq) || !vec_ok(L.bv) || !mat_ok(L.wo) || !vec_ok(L.bo) || !vec_ok(L.ln2_g) ||
            !vec_ok(L.ln2_b) || !mat_ok(L.w1) || !vec_ok(L.b1) || !mat_ok(L.w2) || !vec_ok(L.b2))
            return WH_EINVAL;
    }
    return WH_OK;
}

int run_gemm(const GemmDesc &g, int mode, const DevState *st, cudaStream_t s, int cls = TR_GEMM) {
    trace_begin(cls, s);
    const int rc = gemm_launch(g, mode, ctl_of(st), st->num_sms, s);
    trace_end(cls, s, 2.0 * g.M * (double)g.N * g.K,
              2.0 * ((double)g.M * g.K + (double)g.N * g.K) +
                  (double)g.M * g.N * (mode == GEMM_RESID_F32 ? 8.0 : (mode == GEMM_CONV2 ? 4.0 : 2.0)));
    return rc;
}

GemmDesc gemm(const void *a, int lda, int M, int K, const void *b, int ldb, int N, const float *bias, void *out,
              long long ldo) {
    GemmDesc g;
    std::memset(&g, 0, sizeof(g));
    g.a = a;
    g.lda = lda;
    g.b[0] = g.b[1] = g.b[2] = b;
    g.ldb = ldb;
    g.M = M;
    g.N = N;
    g.K = K;
    g.seg_n = N;
    g.bias[0] = bias;
    g.out = out;
    g.ldo = ldo;
    return g;
}

}  // namespace

void count_launch(int n) { g_launches += n; }

int frontend_ctl(DevCtl *ctl, int *num_sms) {
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    *ctl = ctl_of(st);
    *num_sms = st->num_sms;
    return WH_OK;
}

int device_setup() {
    DevState *st;
    return ensure_device(&st);
}

int device_ctl(DevCtl *ctl, int *num_sms) { return frontend_ctl(ctl, num_sms); }

void trace_begin(int cls, cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_tr_mu);
    if (!g_tr_on) return;
    g_tr_open = tr_event();
    if (g_tr_open) cudaEventRecord(g_tr_open, s);
    (void)cls;
}

void trace_end(int cls, cudaStream_t s, double flops, double bytes) {
    std::lock_guard<std::mutex> lk(g_tr_mu);
    if (!g_tr_on || !g_tr_open) return;
    cudaEvent_t e1 = tr_event();
    if (!e1) return;
    cudaEventRecord(e1, s);
    g_tr.push_back(TraceRec{cls, g_tr_open, e1, flops, bytes});
    g_tr_open = nullptr;
}

}  // namespace wh

using namespace wh;

extern "C" {

const char *wh_strerror(int code) {
    switch (code) {
        case WH_OK: return "WH_OK";
        case WH_EINVAL: return "WH_EINVAL: invalid argument";
        case WH_ENOSPC: return "WH_ENOSPC: workspace too small";
        case WH_ECUDA: return "WH_ECUDA: CUDA call failed";
        case WH_ETIMEOUT: return "WH_ETIMEOUT: a device-side bounded wait ran out";
        case WH_EBOUNDS: return "WH_EBOUNDS: a device-side bounds check fired";
        case WH_ENODEV: return "WH_ENODEV: no usable CUDA device";
    }
    return "WH_E?: unknown code";
}

int64_t wh_launch_count(void) { return g_launches.exchange(0); }

int wh_shutdown(void) {
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        for (DevState &st : g_dev) st = DevState();
    }
    resample_forget();
    return WH_OK;
}

// one word per window (its maximum) and the front-end grid's barrier count
size_t wh_frontend_workspace(int batch) { return batch <= 0 ? 0 : up256(sizeof(uint32_t) * ((size_t)batch + 1)); }

int wh_frontend(const float *pcm, int64_t n, int batch, int n_mels, float *mel, void *workspace, size_t ws_bytes,
                void *stream) {
    if (batch < 0 || batch > 65535 || n < 0 || (n_mels != 80 && n_mels != 128)) return WH_EINVAL;
    if (batch == 0) return WH_OK;
    if (!mel || !workspace || (n > 0 && !pcm)) return WH_EINVAL;
    if (!aligned(mel, 16) || !aligned(workspace, 16)) return WH_EINVAL;
    if (ws_bytes < wh_frontend_workspace(batch)) return WH_ENOSPC;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    trace_begin(TR_FRONTEND, s);
    const int rc = frontend_launch(pcm, n, n, n * batch, batch, n_mels, mel, static_cast<uint32_t *>(workspace),
                                   ctl_of(st), st->num_sms, s);
    const double n_read = (double)(n < 480000 ? n : 480000);
    trace_end(TR_FRONTEND, s, 0.0, batch * (n_read * 4.0 + 3000.0 * n_mels * 4.0));
    return rc;
}

int64_t wh_frontend_windows(int64_t n_total) {
    return n_total <= 0 ? 0 : (n_total + (int64_t)N_FRAMES * 160 - 1) / ((int64_t)N_FRAMES * 160);
}

int wh_frontend_long(const float *pcm, int64_t n_total, int n_mels, float *mel, void *workspace, size_t ws_bytes,
                     void *stream) {
    if (n_total < 0 || (n_mels != 80 && n_mels != 128)) return WH_EINVAL;
    const int64_t windows = wh_frontend_windows(n_total);
    if (windows == 0) return WH_OK;
    if (windows > 65535) return WH_EINVAL;
    if (!pcm || !mel || !workspace || !aligned(pcm, 16) || !aligned(mel, 16) || !aligned(workspace, 16))
        return WH_EINVAL;
    if (ws_bytes < wh_frontend_workspace((int)windows)) return WH_ENOSPC;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t win = (int64_t)N_FRAMES * 160;  // 480000 samples, 30 s
    trace_begin(TR_FRONTEND, s);
    const int rc = frontend_launch(pcm, win, win, n_total, (int)windows, n_mels, mel,
                                   static_cast<uint32_t *>(workspace), ctl_of(st), st->num_sms, s);
    trace_end(TR_FRONTEND, s, 0.0, (double)n_total * 4.0 + (double)windows * N_FRAMES * n_mels * 4.0);
    return rc;
}

int64_t wh_resample_length(int64_t n_in, int rate_in) {
    if (n_in < 0 || !resample_rate_ok(rate_in)) return -1;
    return resample_length(n_in, rate_in);
}

size_t wh_resample_workspace(int rate_in) {
    if (!resample_rate_ok(rate_in)) return 0;
    return up256(resample_workspace(rate_in));
}

int wh_resample(const float *x, int64_t n_in, int batch, int rate_in, float *y, void *workspace, size_t ws_bytes,
                void *stream) {
    if (n_in < 0 || batch < 0 || batch > 65535 || !resample_rate_ok(rate_in)) return WH_EINVAL;
    if (batch == 0 || n_in == 0) return WH_OK;
    if (!x || !y || !workspace || !aligned(x, 4) || !aligned(y, 4) || !aligned(workspace, 16)) return WH_EINVAL;
    if (ws_bytes < wh_resample_workspace(rate_in)) return WH_ENOSPC;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    trace_begin(TR_RESAMPLE, s);
    const int rc = resample_launch(x, n_in, batch, rate_in, y, workspace, st->num_sms, s);
    trace_end(TR_RESAMPLE, s, 0.0, (double)batch * (n_in + resample_length(n_in, rate_in)) * 4.0);
    return rc;
}

size_t wh_encode_workspace(const wh_config *cfg, int batch) {
    if (check_config(cfg) != WH_OK || batch <= 0) return 0;
    return layout(cfg, batch, N_CTX).total;
}

size_t wh_encode_ctx_workspace(const wh_config *cfg, int batch, int n_ctx) {
    if (check_config(cfg) != WH_OK || batch <= 0 || n_ctx < 1 || n_ctx > N_CTX) return 0;
    return layout(cfg, batch, n_ctx).total;
}

int wh_encode_ctx(const float *mel, int batch, int n_ctx, const wh_config *cfg, const wh_weights *w, float *out,
                  void *workspace, size_t ws_bytes, void *stream) {
    if (batch < 0 || n_ctx < 1 || n_ctx > N_CTX) return WH_EINVAL;
    if (int rc = check_config(cfg)) return rc;
    if (batch == 0) return WH_OK;
    if (!mel || !out || !workspace || !aligned(mel, 16) || !aligned(out, 16) || !aligned(workspace, 256))
        return WH_EINVAL;
    if (int rc = check_weights(cfg, w)) return rc;
    const EncLayout L = layout(cfg, batch, n_ctx);
    if (ws_bytes < L.total) return WH_ENOSPC;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int d = cfg->d_model, f = cfg->d_ff, M = cfg->n_mels, H = cfg->n_head;
    const int rows = batch * n_ctx, n_frames = 2 * n_ctx;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *x = reinterpret_cast<float *>(ws + L.x);
    void *xn = ws + L.xn, *qkv = ws + L.qkv, *ao = ws + L.ao, *hb = ws + L.h, *a1 = ws + L.a1;
    void *w1p = ws + L.w1p, *w2p = ws + L.w2p;
    int *sk_tickets = reinterpret_cast<int *>(ws + L.skt);
    int rc;
    const int sk_slots = gemm_sk_slots((long long)rows, d);
    if (cudaMemsetAsync(sk_tickets, 0, gemm_sk_ticket_bytes((long long)rows, d), s) != cudaSuccess) return WH_ECUDA;

    // ---- conv stem over the first 2 n_ctx frames of each window
    trace_begin(TR_STEM_PREP, s);
    if ((rc = pack_conv_weight_launch(w->conv1_w, d, M, w1p, s))) return rc;
    if ((rc = pack_conv_weight_launch(w->conv2_w, d, d, w2p, s))) return rc;
    if ((rc = stem_im2col_launch(mel, batch, M, n_frames, a1, s))) return rc;
    trace_end(TR_STEM_PREP, s, 0.0, (double)batch * n_frames * M * (4.0 + 6.0));
    {
        GemmDesc g = gemm(a1, 3 * M, batch * n_frames, 3 * M, w1p, 3 * M, d, w->conv1_b, qkv, 3LL * d);
        g.rows_per_win = n_frames;
        if ((rc = run_gemm(g, GEMM_CONV1, st, s, TR_GEMM_CONV))) return rc;
    }
    {
        GemmDesc g = gemm(qkv, 3 * d, rows, 3 * d, w2p, 3 * d, d, w->conv2_b, x, d);
        g.pos = w->pos;  // its first n_ctx rows
        g.rows_per_win = n_ctx;
        if ((rc = run_gemm(g, GEMM_CONV2, st, s, TR_GEMM_CONV))) return rc;
    }
    // ---- blocks
    for (int l = 0; l < cfg->n_layer; ++l) {
        const wh_layer_weights &Lw = w->layers[l];
        trace_begin(TR_LAYERNORM, s);
        if ((rc = layernorm_launch(x, rows, d, Lw.ln1_g, Lw.ln1_b, xn, 1, s, false, true))) return rc;
        trace_end(TR_LAYERNORM, s, 0.0, (double)rows * d * 6.0);
        {
            GemmDesc g = gemm(xn, d, rows, d, Lw.wq, d, 3 * d, Lw.bq, qkv, 3LL * d);
            g.b[1] = Lw.wk;
            g.b[2] = Lw.wv;
            g.seg_n = d;
            g.bias[1] = nullptr;  // k_proj has no bias
            g.bias[2] = Lw.bv;
            if ((rc = run_gemm(g, GEMM_BF16, st, s, TR_GEMM_QKV))) return rc;
        }
        trace_begin(TR_ATTN, s);
        if ((rc = attention_launch(qkv, batch, n_ctx, H, ao, ctl_of(st), st->num_sms, s))) return rc;
        trace_end(TR_ATTN, s, 4.0 * batch * (double)n_ctx * n_ctx * d, (double)rows * d * 8.0);
        {
            GemmDesc g = gemm(ao, d, rows, d, Lw.wo, d, d, Lw.bo, x, d);
            g.sk_ws = ws + L.sk;
            g.sk_tickets = sk_tickets;
            g.sk_slots = sk_slots;
            if ((rc = run_gemm(g, GEMM_RESID_F32, st, s, TR_GEMM_OUT))) return rc;
        }
        trace_begin(TR_LAYERNORM, s);
        if ((rc = layernorm_launch(x, rows, d, Lw.ln2_g, Lw.ln2_b, xn, 1, s, false, true))) return rc;
        trace_end(TR_LAYERNORM, s, 0.0, (double)rows * d * 6.0);
        if ((rc = run_gemm(gemm(xn, d, rows, d, Lw.w1, d, f, Lw.b1, hb, f), GEMM_GELU_BF16, st, s, TR_GEMM_FC1)))
            return rc;
        {
            GemmDesc g = gemm(hb, f, rows, f, Lw.w2, f, d, Lw.b2, x, d);
            g.sk_ws = ws + L.sk;
            g.sk_tickets = sk_tickets;
            g.sk_slots = sk_slots;
            if ((rc = run_gemm(g, GEMM_RESID_F32, st, s, TR_GEMM_FC2))) return rc;
        }
    }
    trace_begin(TR_LAYERNORM, s);
    rc = layernorm_launch(x, rows, d, w->lnf_g, w->lnf_b, out, 0, s, false, true);
    trace_end(TR_LAYERNORM, s, 0.0, (double)rows * d * 8.0);
    return rc;
}

int wh_encode(const float *mel, int batch, const wh_config *cfg, const wh_weights *w, float *out, void *workspace,
              size_t ws_bytes, void *stream) {
    return wh_encode_ctx(mel, batch, N_CTX, cfg, w, out, workspace, ws_bytes, stream);
}

size_t wh_prepare_cross_workspace(int batch, int n_ctx, int d_model) {
    if (batch <= 0 || n_ctx < 1 || n_ctx > N_CTX || d_model < 128 || d_model > 2048 || d_model % 128 != 0) return 0;
    return up256((size_t)batch * n_ctx * d_model * 2);
}

int wh_prepare_cross(const float *mem, int batch, int n_ctx, int d_model, int n_layer, const wh_cross_weights *w,
                     wh_bf16 *kv, void *workspace, size_t ws_bytes, void *stream) {
    if (batch < 0 || n_ctx < 1 || n_ctx > N_CTX || n_layer < 0) return WH_EINVAL;
    if (d_model < 128 || d_model > 2048 || d_model % 128 != 0) return WH_EINVAL;
    if (batch == 0 || n_layer == 0) return WH_OK;
    if (!mem || !kv || !workspace || !w || !w->wk || !w->wv || !w->bv) return WH_EINVAL;
    if (!aligned(mem, 16) || !aligned(kv, 16) || !aligned(workspace, 256)) return WH_EINVAL;
    for (int l = 0; l < n_layer; ++l)
        if (!mat_ok(w->wk[l]) || !mat_ok(w->wv[l]) || (w->bv[l] != nullptr && !aligned(w->bv[l], 16)))
            return WH_EINVAL;
    if (ws_bytes < wh_prepare_cross_workspace(batch, n_ctx, d_model)) return WH_ENOSPC;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int d = d_model, rows = batch * n_ctx;
    trace_begin(TR_CROSS_PREP, s);
    int rc = cast_bf16_launch(mem, (long long)rows * d, workspace, s);
    trace_end(TR_CROSS_PREP, s, 0.0, (double)rows * d * 6.0);
    if (rc) return rc;
    for (int l = 0; l < n_layer; ++l) {
        // one GEMM per decoder layer, two output segments: [K | V] = mem [Wk; Wv]^T + [0; bv]
        GemmDesc g = gemm(workspace, d, rows, d, w->wk[l], d, 2 * d, nullptr, kv + (size_t)l * rows * 2 * d, 2LL * d);
        g.b[1] = w->wv[l];
        g.seg_n = d;
        g.bias[1] = w->bv[l];
        if ((rc = run_gemm(g, GEMM_BF16, st, s, TR_GEMM_CROSS))) return rc;
    }
    return WH_OK;
}

size_t wh_decode_attention_workspace(int batch, int n_head, int max_keys) {
    if (batch > 65535 || n_head > 65535 || max_keys > (1 << 30)) return 0;
    return decode_attention_workspace(batch, n_head, max_keys);
}

int wh_decode_attention(const wh_bf16 *q, const wh_bf16 *k, const wh_bf16 *v, int64_t row_stride, int64_t seq_stride,
                        const int *n_keys, int max_keys, int batch, int n_head, wh_bf16 *out, void *workspace,
                        size_t ws_bytes, void *stream) {
    if (batch < 0 || batch > 65535 || n_head < 1 || n_head > 65535 || max_keys < 1 || max_keys > (1 << 30))
        return WH_EINVAL;
    if (row_stride < 64LL * n_head || row_stride % 8 != 0 || seq_stride < 0 || seq_stride % 8 != 0) return WH_EINVAL;
    if (batch == 0) return WH_OK;
    if (!q || !k || !v || !out || !workspace) return WH_EINVAL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(workspace, 256) ||
        (n_keys && !aligned(n_keys, 4)))
        return WH_EINVAL;
    if (ws_bytes < decode_attention_workspace(batch, n_head, max_keys)) return WH_ENOSPC;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    trace_begin(TR_DEC_ATTN, s);
    const int rc = decode_attention_launch(q, k, v, row_stride, seq_stride, n_keys, max_keys, batch, n_head, out,
                                           workspace, ctl_of(st), st->num_sms, s);
    trace_end(TR_DEC_ATTN, s, 4.0 * batch * (double)max_keys * 64.0 * n_head,
              (double)batch * n_head * max_keys * 256.0);
    return rc;
}

int wh_layer_norm(const float *x, int rows, int d, const float *g, const float *b, void *y, int y_bf16,
                  void *stream) {
    if (rows < 0 || d < 64 || d > 2048 || d % 64 != 0) return WH_EINVAL;
    if (rows == 0) return WH_OK;
    if (!x || !g || !b || !y || !aligned(x, 16) || !aligned(g, 16) || !aligned(b, 16) || !aligned(y, 16))
        return WH_EINVAL;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    trace_begin(TR_LAYERNORM, s);
    const int rc = layernorm_launch(x, rows, d, g, b, y, y_bf16, s);
    trace_end(TR_LAYERNORM, s, 0.0, (double)rows * d * (y_bf16 ? 6.0 : 8.0));
    return rc;
}

int wh_linear(const wh_bf16 *a, int rows, int k, const wh_bf16 *w, int n, const float *bias, int epilogue, void *y,
              void *stream) {
    if (rows < 0 || k <= 0 || k % 8 != 0 || n <= 0 || n % 128 != 0) return WH_EINVAL;
    if (epilogue != WH_EPI_BF16 && epilogue != WH_EPI_GELU_BF16 && epilogue != WH_EPI_RESID_F32) return WH_EINVAL;
    if (rows == 0) return WH_OK;
    if (!a || !w || !y || !aligned(a, 16) || !aligned(w, 16) || !aligned(y, 16) || (bias && !aligned(bias, 16)))
        return WH_EINVAL;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    const int mode = epilogue == WH_EPI_BF16 ? GEMM_BF16 : (epilogue == WH_EPI_GELU_BF16 ? GEMM_GELU_BF16 : GEMM_RESID_F32);
    return run_gemm(gemm(a, k, rows, k, w, k, n, bias, y, n), mode, st, static_cast<cudaStream_t>(stream));
}

int wh_attention(const wh_bf16 *qkv, int batch, int n_ctx, int n_head, wh_bf16 *out, void *stream) {
    if (batch < 0 || n_ctx < 1 || n_ctx > N_CTX || n_head < 1 || n_head > 64) return WH_EINVAL;
    if (batch == 0) return WH_OK;
    if (!qkv || !out || !aligned(qkv, 16) || !aligned(out, 16)) return WH_EINVAL;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    trace_begin(TR_ATTN, s);
    const int rc = attention_launch(qkv, batch, n_ctx, n_head, out, ctl_of(st), st->num_sms, s);
    trace_end(TR_ATTN, s, 4.0 * batch * (double)n_ctx * n_ctx * 64 * n_head, (double)batch * n_ctx * n_head * 64 * 8.0);
    return rc;
}

int wh_status(void *stream) {
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return WH_ECUDA;
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return WH_ECUDA;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return WH_ECUDA;
    return v;
}

int wh_selftest_timeout(uint64_t limit_ns, void *stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return WH_EINVAL;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    return selftest_timeout_launch(ctl_of(st, limit_ns), static_cast<cudaStream_t>(stream));
}

}  // extern "C"

struct wh_graph {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

namespace {

// Records what `body` launches on `stream` into an instantiated graph (tracing off meanwhile).
template <typename Body>
int record_graph(cudaStream_t s, wh_graph **graph, Body body) {
    bool tracing;
    {
        std::lock_guard<std::mutex> lk(g_tr_mu);
        tracing = g_tr_on;
        g_tr_on = false;  // no event records inside the recorded pass
    }
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaGetLastError();
        std::lock_guard<std::mutex> lk(g_tr_mu);
        g_tr_on = tracing;
        return WH_ECUDA;
    }
    const int rc = body();
    cudaGraph_t g = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(s, &g);
    {
        std::lock_guard<std::mutex> lk(g_tr_mu);
        g_tr_on = tracing;
    }
    if (rc != WH_OK || ec != cudaSuccess || g == nullptr) {
        if (g) cudaGraphDestroy(g);
        cudaGetLastError();
        return rc != WH_OK ? rc : WH_ECUDA;
    }
    cudaGraphExec_t e = nullptr;
    if (cudaGraphInstantiate(&e, g, 0) != cudaSuccess) {
        cudaGraphDestroy(g);
        cudaGetLastError();
        return WH_ECUDA;
    }
    *graph = new wh_graph{g, e};
    return WH_OK;
}

}  // namespace

extern "C" {

int wh_graph_capture(const float *pcm, int64_t n, int batch, const wh_config *cfg, const wh_weights *w, float *mel,
                     float *out, void *fe_ws, size_t fe_ws_bytes, void *enc_ws, size_t enc_ws_bytes, void *stream,
                     wh_graph **graph) {
    if (!graph || !stream || batch <= 0) return WH_EINVAL;
    *graph = nullptr;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;  // constant tables and kernel set-up, outside the capture
    return record_graph(static_cast<cudaStream_t>(stream), graph, [&]() {
        int rc = wh_frontend(pcm, n, batch, cfg ? cfg->n_mels : 0, mel, fe_ws, fe_ws_bytes, stream);
        if (rc == WH_OK) rc = wh_encode(mel, batch, cfg, w, out, enc_ws, enc_ws_bytes, stream);
        return rc;
    });
}

int wh_graph_capture_encode(const float *mel, int batch, const wh_config *cfg, const wh_weights *w, float *out,
                            void *enc_ws, size_t enc_ws_bytes, void *stream, wh_graph **graph) {
    if (!graph || !stream || batch <= 0) return WH_EINVAL;
    *graph = nullptr;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    return record_graph(static_cast<cudaStream_t>(stream), graph,
                        [&]() { return wh_encode(mel, batch, cfg, w, out, enc_ws, enc_ws_bytes, stream); });
}

int wh_graph_capture_decode(const int *tok, const int *pos, int batch, const wh_dec_config *cfg,
                            const wh_dec_weights *w, wh_bf16 *kcache, wh_bf16 *vcache, const wh_bf16 *cross_kv,
                            int n_ctx, float *logits, int *next_tok, void *workspace, size_t ws_bytes, void *stream,
                            wh_graph **graph) {
    if (!graph || !stream || batch <= 0) return WH_EINVAL;
    *graph = nullptr;
    DevState *st;
    if (int rc = ensure_device(&st)) return rc;
    return record_graph(static_cast<cudaStream_t>(stream), graph, [&]() {
        return wh_decode_step(tok, pos, batch, cfg, w, kcache, vcache, cross_kv, n_ctx, logits, next_tok, workspace,
                              ws_bytes, stream);
    });
}

int wh_graph_launch(wh_graph *graph, void *stream) {
    if (!graph) return WH_EINVAL;
    count_launch();
    return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? WH_OK : WH_ECUDA;
}

int wh_graph_destroy(wh_graph *graph) {
    if (!graph) return WH_EINVAL;
    cudaGraphExecDestroy(graph->exec);
    cudaGraphDestroy(graph->graph);
    delete graph;
    return WH_OK;
}

int wh_trace_enable(int on) {
    std::lock_guard<std::mutex> lk(g_tr_mu);
    g_tr_on = on != 0;
    if (g_tr_on) {
        g_tr.clear();
        g_tr_used = 0;
        g_tr_open = nullptr;
    }
    return WH_OK;
}

int wh_trace_read(wh_trace_stat *out, int max) {
    if (!out || max <= 0) return -WH_EINVAL;
    std::lock_guard<std::mutex> lk(g_tr_mu);
    wh_trace_stat acc[TR_NCLASS];
    std::memset(acc, 0, sizeof(acc));
    for (int c = 0; c < TR_NCLASS; ++c) std::strncpy(acc[c].name, kTraceNames[c], sizeof(acc[c].name) - 1);
    for (const TraceRec &r : g_tr) {
        if (cudaEventSynchronize(r.e1) != cudaSuccess) return -WH_ECUDA;
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, r.e0, r.e1) != cudaSuccess) return -WH_ECUDA;
        acc[r.cls].launches += 1;
        acc[r.cls].total_ms += ms;
        acc[r.cls].flops += r.flops;
        acc[r.cls].bytes += r.bytes;
    }
    int n = 0;
    for (int c = 0; c < TR_NCLASS && n < max; ++c)
        if (acc[c].launches > 0) out[n++] = acc[c];
    return n;
}

}  // extern "C"
