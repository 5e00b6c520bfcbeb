// One-query attention of a decoder step, keys split across blocks with a partial-softmax
// merge ("whisper" package page, "Performance and memory": a decode step has a single query
// per head, so the keys are split across blocks and the blocks' partial softmaxes merged;
// "whisper 0.9.0 API", wh_decode_step: with one query at the end of the sequence the
// self-attention needs no mask, and the cross-attention reads all encoder positions).
//
// For each sequence b and head h:  o = softmax(q k^T / sqrt(64)) v  over the n_keys[b] keys.
//
// Grid (n_head, splits, batch).  A block takes a contiguous range of keys.  Four
// lanes share one key (16 of the 64 dims each, two 16-byte loads of k and of v), so a warp
// covers 8 keys per iteration and every key row is read as whole 32-byte sectors.  Each
// 4-lane group keeps its own running max m, sum l and 16 dims of o (exp2 domain, the 1/8
// scale folded into q); the groups, then the warps, are merged, and the block's partial
// (m, l, o[64]) goes to the workspace (or, with a single split, straight to the output).
// With several splits, the block that finishes last for its (b, h) (an atomic
// ticket; no block waits for another) merges the partials: m = max m_s,
// o = sum_s 2^(m_s - m) o_s / sum_s 2^(m_s - m) l_s.
// HBM-bound: every key and value row is read once; 4 n_keys * 64 bytes per (b, h).
#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

// Grid order: with the head fastest, the blocks that run together read the same key rows
// (all heads of a row are contiguous), so DRAM pages and L2 lines are shared.
constexpr int BLOCKS_PER_SM = 2;   // target blocks per SM over the grid
constexpr int UNROLL = 2;          // key slots in flight per lane group
constexpr int DA_THREADS = 256;
constexpr int DA_WARPS = DA_THREADS / 32;
constexpr int KEYS_PER_ITER = DA_WARPS * 8;   // 32 keys per block iteration
constexpr int PART = 66;                      // floats per partial: m, l, o[64]

struct DecAttnArgs {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k, *v;
    long long row_stride, seq_stride;   // elements
    const int *n_keys;                  // device [batch] or null
    int max_keys, n_head, splits, chunk;
    int *status;                        // per-device status word (WH_EBOUNDS)
    __nv_bfloat16 *out;
    float *part;                        // [batch * n_head * splits][PART]
    int *ticket;                        // [batch * n_head], zero on entry, zero on exit
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// (m, l, o) <- merge of (m, l, o) and (m2, l2, o2), exp2 domain
__device__ __forceinline__ void merge_into(float &m, float &l, float *o, float m2, float l2, const float *o2, int n) {
    const float mn = fmaxf(m, m2);
    const float a = (m == -INFINITY) ? 0.0f : ex2_approx(m - mn);
    const float c = (m2 == -INFINITY) ? 0.0f : ex2_approx(m2 - mn);
    l = l * a + l2 * c;
    for (int i = 0; i < n; ++i) o[i] = o[i] * a + o2[i] * c;
    m = mn;
}

__global__ void __launch_bounds__(DA_THREADS) k_decode_attention(const DecAttnArgs p) {
    const int s = blockIdx.y, h = blockIdx.x, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 2, sub = lane & 3;   // key slot in the warp, 16-dim quarter
    pdl_launch_dependents();
    pdl_wait();
    int nk = p.max_keys;
    if (p.n_keys) {   // a count outside 0 .. max_keys is clamped and reported as WH_EBOUNDS
        const int want = p.n_keys[b];
        nk = min(max(want, 0), p.max_keys);
        if (want != nk && s == 0 && h == 0 && threadIdx.x == 0) atomicCAS(p.status, 0, WH_EBOUNDS);
    }
    const int k0 = s * p.chunk, k1 = min(nk, k0 + p.chunk);

    // q quarter, scaled by log2(e) / 8
    float q[16];
    {
        const uint4 *qp = reinterpret_cast<const uint4 *>(p.q + (long long)b * p.n_head * 64 + h * 64 + 16 * sub);
        bf16x8_to_f32(__ldg(qp), q);
        bf16x8_to_f32(__ldg(qp + 1), q + 8);
        const float sc = 0.125f * 1.4426950408889634f;
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] *= sc;
    }
    const __nv_bfloat16 *kb = p.k + (long long)b * p.seq_stride + h * 64 + 16 * sub;
    const __nv_bfloat16 *vb = p.v + (long long)b * p.seq_stride + h * 64 + 16 * sub;

    float m = -INFINITY, l = 0.0f, o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = 0.0f;

    // UNROLL key slots per lane group in flight: keys t, t + KEYS_PER_ITER, ...  The trip
    // count is uniform across the warp (the shuffles below need every lane); slots past the
    // range skip the update.
    for (int wbase = k0 + warp * 8; wbase < k1; wbase += UNROLL * KEYS_PER_ITER) {
        uint4 kr[UNROLL][2], vr[UNROLL][2];
        bool live[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int t = wbase + grp + u * KEYS_PER_ITER;
            live[u] = t < k1;
            if (live[u]) {
                const uint4 *kp = reinterpret_cast<const uint4 *>(kb + (long long)t * p.row_stride);
                const uint4 *vp = reinterpret_cast<const uint4 *>(vb + (long long)t * p.row_stride);
                kr[u][0] = __ldg(kp);
                kr[u][1] = __ldg(kp + 1);
                vr[u][0] = __ldg(vp);
                vr[u][1] = __ldg(vp + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            float kf[16];
            bf16x8_to_f32(kr[u][0], kf);
            bf16x8_to_f32(kr[u][1], kf + 8);
            float dot = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) dot = fmaf(q[i], kf[i], dot);
            dot += __shfl_xor_sync(0xffffffffu, dot, 1);
            dot += __shfl_xor_sync(0xffffffffu, dot, 2);
            if (!live[u]) continue;   // uniform within the 4-lane group
            float vf[16];
            bf16x8_to_f32(vr[u][0], vf);
            bf16x8_to_f32(vr[u][1], vf + 8);
            const float mn = fmaxf(m, dot);
            const float c = ex2_approx(m - mn);   // m = -inf on the first key: c = 0
            const float e = ex2_approx(dot - mn);
            l = l * c + e;
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = fmaf(o[i], c, e * vf[i]);
            m = mn;
        }
    }

    // merge the 8 key slots of the warp (lanes with the same `sub` hold the same dims)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
        float o2[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) o2[i] = __shfl_xor_sync(0xffffffffu, o[i], off);
        merge_into(m, l, o, m2, l2, o2, 16);
    }
    // merge the warps through shared memory
    __shared__ float sm[DA_WARPS][PART];
    if (grp == 0) {
        if (sub == 0) {
            sm[warp][0] = m;
            sm[warp][1] = l;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) sm[warp][2 + 16 * sub + i] = o[i];
    }
    __syncthreads();
    const long long bh = (long long)b * p.n_head + h;
    if (p.splits == 1) {  // the block saw every key: write the result, no merge
        if (threadIdx.x < 64) {
            float mb = sm[0][0], lb = sm[0][1], ob = sm[0][2 + threadIdx.x];
            for (int w = 1; w < DA_WARPS; ++w)
                merge_into(mb, lb, &ob, sm[w][0], sm[w][1], &sm[w][2 + threadIdx.x], 1);
            p.out[bh * 64 + threadIdx.x] = __float2bfloat16_rn(lb > 0.0f ? ob / lb : 0.0f);
        }
        return;
    }
    float *part = p.part + (bh * p.splits + s) * PART;
    if (threadIdx.x < 64) {  // thread i owns dim i of the block's partial
        float mb = sm[0][0], lb = sm[0][1], ob = sm[0][2 + threadIdx.x];
        for (int w = 1; w < DA_WARPS; ++w) merge_into(mb, lb, &ob, sm[w][0], sm[w][1], &sm[w][2 + threadIdx.x], 1);
        part[2 + threadIdx.x] = ob;
        if (threadIdx.x == 0) {
            part[0] = mb;
            part[1] = lb;
        }
        __threadfence();
    }
    __syncthreads();
    __shared__ int last;
    if (threadIdx.x == 0) last = atomicAdd(p.ticket + bh, 1) == p.splits - 1;
    __syncthreads();
    if (!last) return;
    // the last block of this (b, h): merge every split's partial
    __threadfence();
    if (threadIdx.x < 64) {
        const float *pb = p.part + bh * p.splits * PART;
        float mt = -INFINITY, lt = 0.0f, ot = 0.0f;
        for (int j = 0; j < p.splits; ++j) {
            const float mj = __ldcg(pb + j * PART), lj = __ldcg(pb + j * PART + 1);
            const float oj = __ldcg(pb + j * PART + 2 + threadIdx.x);
            merge_into(mt, lt, &ot, mj, lj, &oj, 1);
        }
        const float r = lt > 0.0f ? ot / lt : 0.0f;   // no keys: zeros
        p.out[bh * 64 + threadIdx.x] = __float2bfloat16_rn(r);
    }
    if (threadIdx.x == 0) p.ticket[bh] = 0;   // ready for the next call
}

}  // namespace

size_t decode_attention_ticket_offset(int batch, int n_head, int max_keys) {
    const size_t max_splits = (size_t)(max_keys + KEYS_PER_ITER - 1) / KEYS_PER_ITER;
    const size_t bh = (size_t)batch * n_head;
    return (bh * max_splits * PART * sizeof(float) + 255) & ~(size_t)255;
}

size_t decode_attention_ticket_bytes(int batch, int n_head) { return (size_t)batch * n_head * sizeof(int); }

size_t decode_attention_workspace(int batch, int n_head, int max_keys) {
    if (batch <= 0 || n_head <= 0 || max_keys <= 0) return 0;
    return decode_attention_ticket_offset(batch, n_head, max_keys) +
           ((decode_attention_ticket_bytes(batch, n_head) + 255) & ~(size_t)255);
}

int decode_attention_launch(const void *q, const void *k, const void *v, long long row_stride, long long seq_stride,
                            const int *n_keys, int max_keys, int batch, int n_head, void *out, void *workspace,
                            const DevCtl &ctl, int num_sms, cudaStream_t s, bool pdl, bool zero_tickets) {
    if (batch <= 0) return WH_OK;
    const long long bh = (long long)batch * n_head;
    // about BLOCKS_PER_SM blocks per SM in total, at least 64 keys per block, chunks a
    // multiple of 32 keys
    long long splits = ((long long)BLOCKS_PER_SM * num_sms + bh - 1) / bh;
    const long long max_by_keys = (max_keys + 63) / 64;
    if (splits > max_by_keys) splits = max_by_keys;
    if (splits < 1) splits = 1;
    int chunk = (int)((max_keys + splits - 1) / splits);
    chunk = (chunk + KEYS_PER_ITER - 1) / KEYS_PER_ITER * KEYS_PER_ITER;
    splits = (max_keys + chunk - 1) / chunk;
    if (splits > 65535 || n_head > 65535) return WH_EINVAL;
    DecAttnArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.v = static_cast<const __nv_bfloat16 *>(v);
    a.row_stride = row_stride;
    a.seq_stride = seq_stride;
    a.n_keys = n_keys;
    a.max_keys = max_keys;
    a.n_head = n_head;
    a.splits = (int)splits;
    a.chunk = chunk;
    a.status = ctl.status;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.part = static_cast<float *>(workspace);
    a.ticket = reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) +
                                       decode_attention_ticket_offset(batch, n_head, max_keys));
    if (zero_tickets && splits > 1 && cudaMemsetAsync(a.ticket, 0, bh * sizeof(int), s) != cudaSuccess)
        return WH_ECUDA;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(n_head, (unsigned)splits, batch);
    lc.blockDim = dim3(DA_THREADS);
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&lc, k_decode_attention, a);
    count_launch();
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

}  // namespace wh
