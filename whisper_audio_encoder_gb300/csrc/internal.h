// Host-side interfaces between the translation units of libwh.so (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace wh {

struct DevCtl;

// ---- GEMM (gemm_tc.cu) -----------------------------------------------------------------
enum GemmMode {
    GEMM_BF16 = 0,        // y bf16 = acc + bias[segment]
    GEMM_GELU_BF16 = 1,   // y bf16 = GELU(acc + bias)
    GEMM_RESID_F32 = 2,   // y f32 += acc + bias
    GEMM_CONV1 = 3,       // GELU(acc + bias) scattered as bf16 into conv2's im2col matrix
    GEMM_CONV2 = 4,       // y f32 = GELU(acc + bias) + pos[row % rows_per_win]
};

struct GemmDesc {
    const void *a; int lda;               // bf16 [M][lda], K columns used
    const void *b[3]; int ldb;            // bf16 [seg_n][ldb] per segment (K columns used)
    int M, N, K, seg_n;                   // N = n_seg * seg_n
    const float *bias[3];                 // per segment, nullable
    void *out; long long ldo;             // output (elements)
    const float *pos;                     // GEMM_CONV2: [rows_per_win][N]
    int rows_per_win;                     // GEMM_CONV1: c1 frames per window; GEMM_CONV2: positions
    // GEMM_RESID_F32, optional (null: whole tiles only): scratch for stream-K with room for
    // sk_slots pair boundaries (gemm_sk_bytes), and sk_slots * 2 * 8 ints that are zero before
    // the first launch (each launch leaves them zero)
    void *sk_ws;
    int *sk_tickets;
    int sk_slots;
};
constexpr int GEMM_SK_SLOTS = 128;   // pair boundaries the scratch holds at most
// Stream-K slots worth keeping for a residual GEMM of M rows and N = ldo columns, and their bytes.
inline int gemm_sk_slots(long long M, int N) {
    const int bn = N % 256 == 0 ? 256 : 128;
    const long long tiles = (M + 255) / 256 * (N / bn) + 1;
    return (int)(tiles < GEMM_SK_SLOTS ? tiles : GEMM_SK_SLOTS);
}
inline size_t gemm_sk_bytes(long long M, int N) {
    return (size_t)gemm_sk_slots(M, N) * 2 * 256 * (N % 256 == 0 ? 256 : 128) * 4;
}
inline size_t gemm_sk_ticket_bytes(long long M, int N) { return (size_t)gemm_sk_slots(M, N) * 2 * 8 * 4; }
// 2-D bf16 TMA descriptor: rows x cols (row stride ld elements), box 64 x box_rows, 128-byte
// swizzle, zero fill outside.  Returns a WH_* code.
int make_tmap_bf16(CUtensorMap *m, const void *ptr, long long rows, int cols, int ld, int box_rows);
// The same for fp32 with a 32-column (128-byte) box.
int make_tmap_f32(CUtensorMap *m, const void *ptr, long long rows, int cols, int ld, int box_rows);

// Returns a WH_* code.  Encodes the tensor maps and launches the persistent tcgen05 kernel.
int gemm_launch(const GemmDesc &g, int mode, const DevCtl &ctl, int num_sms, cudaStream_t s);
// Host-side set-up of every GEMM variant (function attributes, resident-pair counts) on the
// current device, so that later launches do no set-up work (e.g. inside a stream capture).
int gemm_prepare(int num_sms);

// ---- front end (frontend.cu) -------------------------------------------------------------
int frontend_init_tables();   // once per device (current device)
// window b: pcm + b * stride, min(n, total - b * stride) samples
int frontend_launch(const float *pcm, int64_t n, int64_t stride, int64_t total, int batch, int n_mels, float *mel,
                    uint32_t *ws, const DevCtl &ctl, int num_sms, cudaStream_t s);
int frontend_ctl(DevCtl *ctl, int *num_sms);   // the current device's control block and SM count

// ---- other kernels ---------------------------------------------------------------------
// pdl: launched with programmatic stream serialization (may start before the previous kernel
// has finished; waits for it before reading x).  reverse: rows are taken from the last one
// down (after a kernel that stored them in ascending order, its last rows are still in L2).
int layernorm_launch(const float *x, int rows, int d, const float *g, const float *b, void *y, int y_bf16,
                     cudaStream_t s, bool pdl = false, bool reverse = false);
int attention_launch(const void *qkv, int batch, int n_ctx, int n_head, void *out, const DevCtl &ctl,
                     int num_sms, cudaStream_t s);
int attention_prepare();
// windowed-sinc resampling to 16 kHz (resample.cu)
bool resample_rate_ok(int rate_in);
long long resample_length(long long n_in, int rate_in);
size_t resample_workspace(int rate_in);
int resample_launch(const float *x, long long n_in, int batch, int rate_in, float *y, void *table, int num_sms,
                    cudaStream_t s);
int resample_prepare();
void resample_forget();   // drops the per-rate filter normalisers (wh_shutdown)
// one-query attention of a decoder step, keys split across blocks (decode_attention.cu)
size_t decode_attention_workspace(int batch, int n_head, int max_keys);
// pdl: as for layernorm_launch.  zero_tickets = false: the caller guarantees that the merge
// tickets in the workspace (at decode_attention_ticket_offset, decode_attention_ticket_bytes)
// are zero, as every call leaves them.
int decode_attention_launch(const void *q, const void *k, const void *v, long long row_stride, long long seq_stride,
                            const int *n_keys, int max_keys, int batch, int n_head, void *out, void *workspace,
                            const DevCtl &ctl, int num_sms, cudaStream_t s, bool pdl = false,
                            bool zero_tickets = true);
size_t decode_attention_ticket_offset(int batch, int n_head, int max_keys);
size_t decode_attention_ticket_bytes(int batch, int n_head);
// conv1's im2col matrix over the first n_frames (<= 3000) frames of each window's log-mel
int stem_im2col_launch(const float *mel, int batch, int n_mels, int n_frames, void *a1, cudaStream_t s);
// y (bf16) = x (float32), n a multiple of 4, both 16-byte aligned
int cast_bf16_launch(const float *x, long long n, void *y, cudaStream_t s);
int pack_conv_weight_launch(const void *w, int c_out, int c_in, void *wp, cudaStream_t s);
int selftest_timeout_launch(const DevCtl &ctl, cudaStream_t s);

// ---- decoder step (decode_step.cu) ---------------------------------------------------------
int dec_gemm_prepare();   // once per device: shared-memory attributes of the step's GEMMs

// ---- per-device set-up (wh_api.cu): constant tables and status word, once per device ----
int device_setup();
int device_ctl(DevCtl *ctl, int *num_sms);     // the current device's control block and SM count

// ---- tracing (wh_api.cu) ------------------------------------------------------------------
// Kernel classes for the per-kernel timing.
enum TraceClass {
    TR_FRONTEND = 0, TR_STEM_PREP, TR_GEMM, TR_ATTN, TR_LAYERNORM,
    TR_GEMM_CONV, TR_GEMM_QKV, TR_GEMM_OUT, TR_GEMM_FC1, TR_GEMM_FC2, TR_CROSS_PREP, TR_GEMM_CROSS, TR_DEC_ATTN, TR_RESAMPLE,
    TR_DEC_GEMM, TR_DEC_OTHER, TR_NCLASS
};
void trace_begin(int cls, cudaStream_t s);
void trace_end(int cls, cudaStream_t s, double flops, double bytes);
void count_launch(int n = 1);

}  // namespace wh
