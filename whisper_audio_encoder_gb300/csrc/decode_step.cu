// One decoder step for a batch of sequences ("whisper 0.9.0 API", model.nu, wh_decode_step:
// token tok at position pos with everything before it already in the KV cache, the logits
// left on the device; wk_addv_row: the stored position row is added; setrow: the token's
// key and value are written into the cache; wh_argmax: greedy decoding on the device.
// "How Audio Becomes Words", "The Full Stitched Circuit": each decoder block is causal
// self-attention, cross-attention into the encoder memory and a feed-forward, each behind
// its own LayerNorm and added to the residual; a final norm and the output projection
// through the token embedding follow.)
//
// Per step: k_dec_embed, then per layer LN -> QKV (q out, k / v appended at row pos of the
// caches) -> one-query self-attention over rows 0..pos -> out_proj + residual -> LN -> cross
// q -> one-query cross-attention over the layer's cached K/V -> cross out + residual -> LN ->
// fc1 + GELU -> fc2 + residual; final LN -> logits (+ argmax) -> next token.
//
// k_dec_gemm: the step's dense layers have one row per sequence (a few to a few hundred), so
// they stream their weights once and are bound by HBM.  On the tensor cores the weights are
// the M operand: a CTA computes D[128 features][B tokens] = W[n0 .. n0+127][K] X[B][K]^T with
// tcgen05.mma (M = 128, N = B rounded up to 16, K = 16), both operands K-major from a TMA ring,
// the accumulator in TMEM (lane = feature, column = token).  K is split across CTAs so that
// every SM streams weights: the splits of a tile are one thread-block cluster, each CTA stages
// its partial tile in shared memory, and after a cluster barrier each CTA adds the partials of
// its slice of the tile in split order through distributed shared memory and applies the
// epilogue -- no partial sums go through global memory, and the result does not depend on
// timing.  Launched with programmatic stream serialization: the weight stream starts while
// the previous kernel is still running; only the activations wait for it.
#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

constexpr int SK_THREADS = 192;   // warp 0 TMA, warp 1 TMEM + MMA, warps 2..5 epilogue
constexpr int SK_STAGES = 4;
constexpr int SK_BK = 64;
constexpr int SK_W_BYTES = 128 * SK_BK * 2;   // one k-block of 128 weight rows
constexpr int SK_MAX_SPLITS = 8;    // splits of one tile form a (portable) cluster
constexpr int SK_MAX_B = 256;

enum SkMode { SK_QKV = 0, SK_BF16 = 1, SK_GELU = 2, SK_RESID = 3, SK_LOGITS = 4 };

struct SkArgs {
    int N, seg_n, num_kb, kb_per, B, B_pad, x_bytes, stage_bytes, tmem_cols;
    // LayerNorm fused in front (xf != nullptr): the operand X is LN(xf) over K = d columns,
    // built by the epilogue warps in shared memory at x_off instead of loaded by TMA
    const float *xf, *ln_g, *ln_b;
    int K, x_off, bar_off;
    const float *bias[3];
    void *out[3];
    int cap;                    // SK_QKV: cache rows per sequence
    const int *pos;             // SK_QKV: cache row of each sequence (already in range)
    unsigned long long *amax;   // SK_LOGITS: per-sequence (logit key, ~index), zero on entry
    DevCtl ctl;
};
struct SkMaps {
    CUtensorMap w[3];
};

// Order-preserving float -> uint32 (larger float, larger key).
__device__ __forceinline__ uint32_t ord_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// The finished value of output feature n for sequence b.
template <int MODE>
__device__ __forceinline__ void sk_finish(const SkArgs &p, int b, int n, float bias, float v,
                                          unsigned long long &best) {
    v += bias;
    if constexpr (MODE == SK_QKV) {
        const int seg = n / p.seg_n, nin = n - seg * p.seg_n;
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(seg == 0 ? p.out[0] : (seg == 1 ? p.out[1] : p.out[2]));
        const long long row = seg == 0 ? b : (long long)b * p.cap + __ldg(p.pos + b);
        o[row * p.seg_n + nin] = __float2bfloat16_rn(v);
    } else if constexpr (MODE == SK_BF16 || MODE == SK_GELU) {
        if constexpr (MODE == SK_GELU) v = gelu_erf(v);
        static_cast<__nv_bfloat16 *>(p.out[0])[(long long)b * p.N + n] = __float2bfloat16_rn(v);
    } else if constexpr (MODE == SK_RESID) {
        float *x = static_cast<float *>(p.out[0]) + (long long)b * p.N + n;
        *x += v;
    } else {  // SK_LOGITS
        if (n < p.N) {
            static_cast<float *>(p.out[0])[(long long)b * p.N + n] = v;
            best = ((unsigned long long)ord_key(v) << 32) | (unsigned long long)(0xffffffffu - (uint32_t)n);
        } else {
            best = 0ull;
        }
    }
}

// Largest key over the warp (the logit, then the lowest index).
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

template <int MODE>
__global__ void __launch_bounds__(SK_THREADS) k_dec_gemm(const __grid_constant__ SkMaps tw,
                                                         const __grid_constant__ CUtensorMap tx, const SkArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.bar_off);
    uint64_t *empty = full + SK_STAGES;
    uint64_t *accf = empty + SK_STAGES;
    uint64_t *drain = accf + 1;
    uint64_t *x_ready = drain + 1;      // LN-fused operand written (4 epilogue warps)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(x_ready + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ int epi_fail;
    __shared__ unsigned long long cta_best[SK_MAX_B];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, split = blockIdx.y, splits = gridDim.y;
    const int n0 = tile * 128, seg = n0 / p.seg_n, nin0 = n0 - seg * p.seg_n;
    const int kb0 = split * p.kb_per, kb1 = min(p.num_kb, kb0 + p.kb_per);
    const CUtensorMap *wmap = seg == 0 ? &tw.w[0] : (seg == 1 ? &tw.w[1] : &tw.w[2]);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SK_STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(accf, 1);
        mbar_init(drain, 1);
        mbar_init(x_ready, 4);
        *abort_flag = 0;
        epi_fail = 0;
        fence_mbar_init();
        tma_prefetch_desc(wmap);
        tma_prefetch_desc(&tx);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    pdl_launch_dependents();   // the next kernel may start its own weight stream now
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        // The weights do not depend on earlier kernels: the first ring's worth is requested
        // before waiting for the previous kernel, whose output (the activations x) follows.
        const int pre = kb1 - kb0 < SK_STAGES ? kb1 - kb0 : SK_STAGES;
        for (int i = 0; i < pre; ++i) {
            mbar_arrive_expect_tx(full + i, (uint32_t)(SK_W_BYTES + p.x_bytes));
            tma_load_2d(smem + i * p.stage_bytes, wmap, full + i, (kb0 + i) * SK_BK, nin0);
        }
        pdl_wait();
        if (p.xf == nullptr)
            for (int i = 0; i < pre; ++i)
                tma_load_2d(smem + i * p.stage_bytes + SK_W_BYTES, &tx, full + i, (kb0 + i) * SK_BK, 0);
        int stage = pre % SK_STAGES;
        uint32_t phase = pre == SK_STAGES ? 1u : 0u, issued = (1u << pre) - 1u, last_parity = 0;
        for (int kb = kb0 + pre; kb < kb1; ++kb) {
            if (*abort_flag || !mbar_wait(empty + stage, phase ^ 1u, p.ctl)) {
                *abort_flag = 1;
                break;
            }
            uint8_t *sw = smem + stage * p.stage_bytes;
            mbar_arrive_expect_tx(full + stage, (uint32_t)(SK_W_BYTES + p.x_bytes));
            tma_load_2d(sw, wmap, full + stage, kb * SK_BK, nin0);
            if (p.xf == nullptr) tma_load_2d(sw + SK_W_BYTES, &tx, full + stage, kb * SK_BK, 0);
            issued |= 1u << stage;
            last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == SK_STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // no copy of this CTA may still be in flight when it leaves
        for (int s = 0; s < SK_STAGES; ++s)
            if ((issued >> s) & 1u) mbar_wait(full + s, (last_parity >> s) & 1u, p.ctl);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc = idesc_bf16_f32(128, p.B_pad);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = p.xf == nullptr || (!*abort_flag && mbar_wait(x_ready, 0, p.ctl));
        const uint32_t xr = smem_u32(smem + p.x_off);
        for (int kb = kb0; ok && kb < kb1; ++kb) {
            if (*abort_flag || !mbar_wait(full + stage, phase, p.ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * p.stage_bytes);
            const uint64_t ad = sdesc_sw128(sa);
            const uint64_t bd = sdesc_sw128(p.xf ? xr + (uint32_t)((kb - kb0) * p.B_pad * 128) : sa + SK_W_BYTES);
#pragma unroll
            for (int k = 0; k < SK_BK / 16; ++k)
                umma_bf16(tmem_base, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
                          (kb > kb0 || k > 0) ? 1u : 0u);
            umma_commit(empty + stage);
            if (++stage == SK_STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) *abort_flag = 1;
        umma_commit(ok ? accf : drain);
        if (!ok) mbar_wait(drain, 0, p.ctl);   // every MMA issued so far has completed
    } else if (warp >= 2) {
        // ---------------- epilogue: feature n = n0 + 32 q + lane, every sequence ----------------
        const int q = warp & 3, n = n0 + 32 * q + lane;
        if (p.xf != nullptr) {
            // LayerNorm in front (eps 1e-5, biased variance): the epilogue warps write this
            // split's k-blocks of bf16 LN(x) in the 128-byte-swizzled K-major layout the MMA
            // reads; rows B .. B_pad-1 are zero.
            pdl_wait();
            const int kbs = kb1 - kb0, pad_rows = p.B_pad - p.B;
            uint8_t *xs = smem + p.x_off;
            for (int i = threadIdx.x - 64; i < kbs * pad_rows * 8; i += 128) {
                const int kk = i / (pad_rows * 8), rem = i - kk * pad_rows * 8;
                *reinterpret_cast<uint4 *>(xs + kk * p.B_pad * 128 + (p.B + (rem >> 3)) * 128 + (rem & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            // Each warp normalises rows b = w, w + 4, ...: the row in registers (16-byte loads),
            // mean then centred variance, then this split's k-blocks written as bf16.
            const int ew = warp - 2, nv = p.K >> 7;   // float4 per lane
            for (int b = ew; b < p.B; b += 4) {
                const float4 *xrow = reinterpret_cast<const float4 *>(p.xf + (long long)b * p.K);
                float4 v[16];
                float s0 = 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (i < nv) {
                        v[i] = __ldcg(xrow + i * 32 + lane);
                        s0 += (v[i].x + v[i].y) + (v[i].z + v[i].w);
                    }
                const float mean = warp_sum(s0) / (float)p.K;
                float q0 = 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (i < nv) {
                        const float a = v[i].x - mean, c = v[i].y - mean, d2 = v[i].z - mean, e = v[i].w - mean;
                        q0 = fmaf(a, a, fmaf(c, c, fmaf(d2, d2, fmaf(e, e, q0))));
                    }
                const float rstd = 1.0f / sqrtf(warp_sum(q0) / (float)p.K + 1e-5f);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (i < nv) {
                        const int k = 4 * (i * 32 + lane), kb = k >> 6;
                        if (kb >= kb0 && kb < kb1) {
                            const float4 gg = __ldg(reinterpret_cast<const float4 *>(p.ln_g + k));
                            const float4 bb = __ldg(reinterpret_cast<const float4 *>(p.ln_b + k));
                            const uint2 w = make_uint2(pack_bf16((v[i].x - mean) * rstd * gg.x + bb.x,
                                                                 (v[i].y - mean) * rstd * gg.y + bb.y),
                                                       pack_bf16((v[i].z - mean) * rstd * gg.z + bb.z,
                                                                 (v[i].w - mean) * rstd * gg.w + bb.w));
                            const int ch = (k & 63) >> 3;
                            *reinterpret_cast<uint2 *>(xs + (kb - kb0) * p.B_pad * 128 + b * 128 +
                                                       ((ch ^ (b & 7)) << 4) + ((k & 7) >> 2) * 8) = w;
                        }
                    }
            }
            fence_proxy_async_smem();   // the tensor core reads what this warp wrote
            __syncwarp();
            if (lane == 0) mbar_arrive(x_ready);
        }
        if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(accf, 0, p.ctl)) && lane == 0) epi_fail = 1;
        float bias = 0.0f;
        if (MODE != SK_LOGITS && splits == 1) {
            const int sg = n / p.seg_n;
            const float *bp = sg == 0 ? p.bias[0] : (sg == 1 ? p.bias[1] : p.bias[2]);
            if (bp != nullptr) bias = __ldg(bp + (n - sg * p.seg_n));
        }
        if (MODE == SK_LOGITS)
            for (int b = threadIdx.x - 64; b < p.B; b += 128) cta_best[b] = 0ull;
        epi_bar();
        // one verdict for all four epilogue warps, so that they all reach the same barriers
        const bool ok = epi_fail == 0;
        if (!ok) *abort_flag = 1;
        pdl_wait();   // earlier kernels' outputs (x, the cache rows) are complete and visible
        if (ok) {
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16);
            float *P = reinterpret_cast<float *>(smem);   // the ring is free once the MMAs are done
            for (int c = 0; c < p.B_pad; c += 16) {
                uint32_t r[16];
                tmem_ld16(tbase + (uint32_t)c, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int b = c + j;
                    if (b >= p.B) break;
                    const float v = __uint_as_float(r[j]);
                    if (splits > 1) {
                        P[b * 128 + 32 * q + lane] = v;   // this split's partial, [token][feature]
                    } else {
                        unsigned long long best = 0ull;
                        sk_finish<MODE>(p, b, n, bias, v, best);
                        if constexpr (MODE == SK_LOGITS) {
                            best = warp_max_u64(best);
                            if (lane == 0) atomicMax(cta_best + b, best);
                        }
                    }
                }
            }
        }
        if (MODE == SK_LOGITS) {
            epi_bar();
            for (int b = threadIdx.x - 64; b < p.B; b += 128)
                if (cta_best[b] != 0ull) atomicMax(p.amax + b, cta_best[b]);
        }
    }
    tc_fence_before();
    if (MODE != SK_LOGITS && splits > 1) {
        // The splits of this tile are one cluster.  Once every CTA's partial is in its shared
        // memory, CTA r adds, for its slice of the tile's features, the partials of all splits
        // in split order (read through distributed shared memory) and finishes them.  Every
        // thread of every CTA of the cluster reaches both cluster barriers on every path.
        cluster_sync();
        pdl_wait();
        if (!*abort_flag) {
            const int per = (128 + splits - 1) / splits, f0 = split * per;
            const int len = min(128, f0 + per) - f0;
            const uint32_t pl = smem_u32(smem);
            uint32_t peer[SK_MAX_SPLITS];
#pragma unroll
            for (int r = 0; r < SK_MAX_SPLITS; ++r) peer[r] = r < splits ? mapa_shared(smem, (uint32_t)r) : pl;
            for (int i = threadIdx.x; i < len * p.B; i += SK_THREADS) {
                const int b = i / len, nl = f0 + (i - b * len), nn = n0 + nl;
                const uint32_t off = (uint32_t)(b * 128 + nl) * 4u;
                float pv[SK_MAX_SPLITS];
#pragma unroll
                for (int r = 0; r < SK_MAX_SPLITS; ++r) {
                    pv[r] = 0.0f;
                    if (r < splits) asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(pv[r]) : "r"(peer[r] + off));
                }
                float v = 0.0f;
#pragma unroll
                for (int r = 0; r < SK_MAX_SPLITS; ++r)
                    if (r < splits) v += pv[r];
                const int sg = nn / p.seg_n;
                const float *bp = sg == 0 ? p.bias[0] : (sg == 1 ? p.bias[1] : p.bias[2]);
                unsigned long long best = 0ull;
                sk_finish<MODE>(p, b, nn, bp != nullptr ? __ldg(bp + (nn - sg * p.seg_n)) : 0.0f, v, best);
            }
        }
        cluster_sync();   // no CTA leaves while a peer may still read its partial
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
    }
}

// x[b] = tok_embd[tok[b]] + dec_pos[pos[b]] (fp32), the cache row and self-attention key count
// of every sequence, and the argmax keys cleared.  A token or position outside its table is
// clamped into it and reported as WH_EBOUNDS: nothing outside the tables or caches is read or
// written.
__global__ void __launch_bounds__(256) k_dec_embed(const int *__restrict__ tok, const int *__restrict__ pos,
                                                   const __nv_bfloat16 *__restrict__ emb,
                                                   const float *__restrict__ dpos, int d, int n_vocab, int cap,
                                                   float *__restrict__ x, int *__restrict__ pos_c,
                                                   int *__restrict__ n_self, unsigned long long *__restrict__ amax,
                                                   int *status) {
    const int b = blockIdx.x;
    const int t_in = __ldg(tok + b), p_in = __ldg(pos + b);
    const int t = min(max(t_in, 0), n_vocab - 1), ps = min(max(p_in, 0), cap - 1);
    if (threadIdx.x == 0) {
        if (t != t_in || ps != p_in) atomicCAS(status, 0, WH_EBOUNDS);
        pos_c[b] = ps;
        n_self[b] = ps + 1;
        amax[b] = 0ull;
    }
    const uint4 *e = reinterpret_cast<const uint4 *>(emb + (long long)t * d);
    const float4 *pp = reinterpret_cast<const float4 *>(dpos + (long long)ps * d);
    float4 *xo = reinterpret_cast<float4 *>(x + (long long)b * d);
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
        const uint4 u = __ldg(e + i);
        const float4 p0 = __ldg(pp + 2 * i), p1 = __ldg(pp + 2 * i + 1);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        float f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = __uint_as_float(w[j] << 16);
            f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
        }
        xo[2 * i] = make_float4(f[0] + p0.x, f[1] + p0.y, f[2] + p0.z, f[3] + p0.w);
        xo[2 * i + 1] = make_float4(f[4] + p1.x, f[5] + p1.y, f[6] + p1.z, f[7] + p1.w);
    }
}

__global__ void k_dec_argmax_out(const unsigned long long *__restrict__ amax, int batch, int *__restrict__ next) {
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < batch; b += gridDim.x * blockDim.x)
        next[b] = (int)(0xffffffffu - (uint32_t)(amax[b] & 0xffffffffull));
}

int sk_b_pad(int batch) { return (batch + 15) / 16 * 16; }
int sk_stage_bytes(int b_pad) { return SK_W_BYTES + (b_pad * 128 + 1023) / 1024 * 1024; }
int sk_smem_bytes(int b_pad) { return SK_STAGES * sk_stage_bytes(b_pad) + 1024 + 128; }

template <int MODE>
int sk_set_attr() {
    return cudaFuncSetAttribute(k_dec_gemm<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                sk_smem_bytes(SK_MAX_B)) == cudaSuccess
               ? WH_OK
               : WH_ECUDA;
}

}  // namespace

int dec_gemm_prepare() {
    return sk_set_attr<SK_QKV>() | sk_set_attr<SK_BF16>() | sk_set_attr<SK_GELU>() | sk_set_attr<SK_RESID>() |
           sk_set_attr<SK_LOGITS>();
}

// y = epilogue(x[batch][K] w[N][K]^T + bias) for one of the SkMode epilogues.  w may be up to
// three segments of seg_n rows (QKV); N = segments x seg_n, or any N for the logits.
// With xf given, X = LN(xf; ln_g, ln_b) is built inside the kernel (x is not read); if that
// layout does not fit in shared memory, WH_ENOSPC is returned before anything is launched.
int dec_gemm_launch(int mode, const void *x, const float *xf, const float *ln_g, const float *ln_b, int batch,
                    int K, const void *const w[3], int seg_n, int N, const float *const bias[3], void *const out[3],
                    int cap, const int *pos, unsigned long long *amax, const DevCtl &ctl, int num_sms,
                    cudaStream_t s) {
    if (batch < 1 || batch > SK_MAX_B || K < 8 || K % 8 != 0 || N < 1 || seg_n < 1) return WH_EINVAL;
    if (mode != SK_LOGITS && (seg_n % 128 != 0 || N % seg_n != 0 || N / seg_n > 3)) return WH_EINVAL;
    const int b_pad = sk_b_pad(batch);
    SkArgs a;
    a.N = N;
    a.seg_n = mode == SK_LOGITS ? N : seg_n;
    a.num_kb = (K + SK_BK - 1) / SK_BK;
    a.B = batch;
    a.B_pad = b_pad;
    const bool ln_in = xf != nullptr;
    if (ln_in && (K % 128 != 0 || K > 2048)) return WH_EINVAL;
    a.x_bytes = ln_in ? 0 : b_pad * 128;
    a.stage_bytes = ln_in ? SK_W_BYTES : sk_stage_bytes(b_pad);
    a.xf = xf;
    a.ln_g = ln_g;
    a.ln_b = ln_b;
    a.K = K;
    a.tmem_cols = b_pad <= 32 ? 32 : (b_pad <= 64 ? 64 : (b_pad <= 128 ? 128 : 256));
    for (int i = 0; i < 3; ++i) {
        a.bias[i] = bias ? bias[i] : nullptr;
        a.out[i] = out[i];
    }
    a.cap = cap;
    a.pos = pos;
    a.amax = amax;
    a.ctl = ctl;
    SkMaps tw;
    const int nseg = mode == SK_LOGITS ? 1 : N / seg_n;
    for (int i = 0; i < 3; ++i)
        if (int rc = make_tmap_bf16(&tw.w[i], w[i < nseg ? i : 0], a.seg_n, K, K, 128)) return rc;
    CUtensorMap tx = tw.w[0];   // placeholder when the operand is built in the kernel
    if (!ln_in)
        if (int rc = make_tmap_bf16(&tx, x, batch, K, K, b_pad)) return rc;
    const int tiles = (N + 127) / 128;
    // split K so that about one CTA per SM streams weights; the splits of a tile form a
    // cluster of at most SK_MAX_SPLITS CTAs, and every split gets >= 1 k-block
    int splits = 1;
    if (mode != SK_LOGITS) {
        splits = (num_sms + tiles / 2) / tiles;
        splits = splits < 1 ? 1 : (splits > SK_MAX_SPLITS ? SK_MAX_SPLITS : splits);
        splits = splits > a.num_kb ? a.num_kb : splits;
    }
    a.kb_per = (a.num_kb + splits - 1) / splits;
    splits = (a.num_kb + a.kb_per - 1) / a.kb_per;
    if (tiles > 2147483647 / 128) return WH_EINVAL;
    // shared memory: the weight ring (with the TMA-loaded X per stage unless LN is fused), the
    // LN-built X of this split's k-blocks, the barriers, and slack for 1024-byte alignment
    // (after the MMAs the split's partial tile, B x 128 fp32, is staged from offset 0 for the
    // cluster reduction: the barriers must lie beyond it too)
    a.x_off = SK_STAGES * a.stage_bytes;
    a.bar_off = a.x_off + (ln_in ? a.kb_per * b_pad * 128 : 0);
    if (splits > 1 && a.bar_off < batch * 128 * 4) a.bar_off = batch * 128 * 4;
    const int smem = a.bar_off + 128 + 1024;
    if (smem > sk_smem_bytes(SK_MAX_B)) return WH_ENOSPC;
    cudaError_t e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(tiles, splits);
    lc.blockDim = dim3(SK_THREADS);
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = splits;
    attr[1].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = splits > 1 ? 2 : 1;
    switch (mode) {
        case SK_QKV: e = cudaLaunchKernelEx(&lc, k_dec_gemm<SK_QKV>, tw, tx, a); break;
        case SK_BF16: e = cudaLaunchKernelEx(&lc, k_dec_gemm<SK_BF16>, tw, tx, a); break;
        case SK_GELU: e = cudaLaunchKernelEx(&lc, k_dec_gemm<SK_GELU>, tw, tx, a); break;
        case SK_RESID: e = cudaLaunchKernelEx(&lc, k_dec_gemm<SK_RESID>, tw, tx, a); break;
        case SK_LOGITS: e = cudaLaunchKernelEx(&lc, k_dec_gemm<SK_LOGITS>, tw, tx, a); break;
        default: return WH_EINVAL;
    }
    count_launch();
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

int dec_embed_launch(const int *tok, const int *pos, const void *emb, const float *dpos, int d, int n_vocab, int cap,
                     int batch, float *x, int *pos_c, int *n_self, unsigned long long *amax, const DevCtl &ctl,
                     cudaStream_t s) {
    k_dec_embed<<<batch, 256, 0, s>>>(tok, pos, static_cast<const __nv_bfloat16 *>(emb), dpos, d, n_vocab, cap, x,
                                      pos_c, n_self, amax, ctl.status);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

int dec_argmax_launch(const unsigned long long *amax, int batch, int *next, cudaStream_t s) {
    k_dec_argmax_out<<<(batch + 255) / 256, 256, 0, s>>>(amax, batch, next);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

}  // namespace wh

// ---------------------------------------------------------------------------------------
// wh_decode_step: argument checks, workspace layout and the step's launch sequence
// ---------------------------------------------------------------------------------------
namespace wh {
namespace {

constexpr int DEC_MAX_CROSS = 1500;   // encoder positions

size_t up256d(size_t x) { return (x + 255) & ~(size_t)255; }

struct DecLayout {
    size_t x, xn, q, ao, h, pos_c, n_self, amax, da_self, da_cross, total;
};

DecLayout dec_layout(const wh_dec_config *c, int batch) {
    const size_t B = batch, d = c->d_model, f = c->d_ff;
    DecLayout L;
    size_t off = 0;
    L.x = off;      off += up256d(B * d * 4);
    L.xn = off;     off += up256d(B * d * 2);
    L.q = off;      off += up256d(B * d * 2);
    L.ao = off;     off += up256d(B * d * 2);
    L.h = off;      off += up256d(B * f * 2);
    L.pos_c = off;  off += up256d(B * 4);
    L.n_self = off; off += up256d(B * 4);
    L.amax = off;   off += up256d(B * 8);
    // one region each for the self- and the cross-attention, so that each keeps its merge
    // tickets zero between calls
    L.da_self = off;  off += up256d(decode_attention_workspace(batch, c->n_head, c->n_text_ctx));
    L.da_cross = off; off += up256d(decode_attention_workspace(batch, c->n_head, DEC_MAX_CROSS));
    L.total = off;
    return L;
}

int check_dec_config(const wh_dec_config *c) {
    if (!c) return WH_EINVAL;
    if (c->d_model < 128 || c->d_model > 2048 || c->d_model % 128 != 0) return WH_EINVAL;
    if (c->n_head < 1 || c->d_model != 64 * c->n_head) return WH_EINVAL;
    if (c->n_layer < 0 || c->d_ff < 128 || c->d_ff % 128 != 0 || c->d_ff > 16384) return WH_EINVAL;
    if (c->n_vocab < 1 || c->n_vocab > (1 << 24) || c->n_text_ctx < 1 || c->n_text_ctx > 65536) return WH_EINVAL;
    return WH_OK;
}

bool al(const void *p, size_t a) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_dec_weights(const wh_dec_config *c, const wh_dec_weights *w) {
    if (!w || !al(w->tok_embd, 16) || !al(w->pos, 16) || !al(w->lnf_g, 16) || !al(w->lnf_b, 16)) return WH_EINVAL;
    if (c->n_layer > 0 && !w->layers) return WH_EINVAL;
    for (int l = 0; l < c->n_layer; ++l) {
        const wh_dec_layer_weights &L = w->layers[l];
        const void *need[] = {L.ln1_g, L.ln1_b, L.wq, L.wk, L.wv, L.bq, L.bv, L.wo, L.bo, L.lnx_g, L.lnx_b,
                              L.xwq, L.xbq, L.xwo, L.xbo, L.ln2_g, L.ln2_b, L.w1, L.b1, L.w2, L.b2};
        for (const void *p : need)
            if (!al(p, 16)) return WH_EINVAL;
    }
    return WH_OK;
}

}  // namespace
}  // namespace wh

using namespace wh;

extern "C" size_t wh_decode_step_workspace(const wh_dec_config *cfg, int batch) {
    if (check_dec_config(cfg) != WH_OK || batch < 1 || batch > SK_MAX_B) return 0;
    return dec_layout(cfg, batch).total;
}

extern "C" int wh_decode_step(const int *tok, const int *pos, int batch, const wh_dec_config *cfg,
                              const wh_dec_weights *w, wh_bf16 *kcache, wh_bf16 *vcache, const wh_bf16 *cross_kv,
                              int n_ctx, float *logits, int *next_tok, void *workspace, size_t ws_bytes,
                              void *stream) {
    if (int rc = check_dec_config(cfg)) return rc;
    if (batch < 0 || batch > SK_MAX_B || n_ctx < 1 || n_ctx > DEC_MAX_CROSS) return WH_EINVAL;
    if (batch == 0) return WH_OK;
    if (!al(tok, 4) || !al(pos, 4) || !al(logits, 16) || !al(workspace, 256) || (next_tok && !al(next_tok, 4)))
        return WH_EINVAL;
    if (cfg->n_layer > 0 && (!al(kcache, 16) || !al(vcache, 16) || !al(cross_kv, 16))) return WH_EINVAL;
    if (int rc = check_dec_weights(cfg, w)) return rc;
    const DecLayout L = dec_layout(cfg, batch);
    if (ws_bytes < L.total) return WH_ENOSPC;
    DevCtl ctl;
    int num_sms = 0;
    if (int rc = device_ctl(&ctl, &num_sms)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int d = cfg->d_model, f = cfg->d_ff, H = cfg->n_head, cap = cfg->n_text_ctx, V = cfg->n_vocab;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *x = reinterpret_cast<float *>(ws + L.x);
    void *xn = ws + L.xn, *q = ws + L.q, *ao = ws + L.ao, *hb = ws + L.h;
    int *pos_c = reinterpret_cast<int *>(ws + L.pos_c), *n_self = reinterpret_cast<int *>(ws + L.n_self);
    unsigned long long *amax = reinterpret_cast<unsigned long long *>(ws + L.amax);
    uint8_t *da_self = ws + L.da_self, *da_cross = ws + L.da_cross;
    const size_t layer_cache = (size_t)batch * cap * d;
    const size_t layer_cross = (size_t)batch * n_ctx * 2 * d;
    int rc;

    trace_begin(TR_DEC_OTHER, s);
    // every merge ticket of the step starts at zero (each launch leaves its own at zero)
    const size_t da_tickets = decode_attention_ticket_bytes(batch, H);
    if (cudaMemsetAsync(da_self + decode_attention_ticket_offset(batch, H, cap), 0, da_tickets, s) != cudaSuccess ||
        cudaMemsetAsync(da_cross + decode_attention_ticket_offset(batch, H, n_ctx), 0, da_tickets, s) != cudaSuccess)
        return WH_ECUDA;
    rc = dec_embed_launch(tok, pos, w->tok_embd, w->pos, d, V, cap, batch, x, pos_c, n_self, amax, ctl, s);
    trace_end(TR_DEC_OTHER, s, 0.0, (double)batch * d * 10.0);
    if (rc) return rc;

    // A dense layer; with g given, its input is LN(x; g, b), fused into the GEMM when the
    // normalised operand fits in shared memory, else a LayerNorm launch writes xn first.
    auto gemm = [&](int mode, const float *g, const float *b, const void *a, int K, const void *w0, const void *w1,
                    const void *w2, int seg_n, int N, const float *b0, const float *b1, const float *b2, void *o0,
                    void *o1, void *o2) {
        const void *wv[3] = {w0, w1 ? w1 : w0, w2 ? w2 : w0};
        const float *bv[3] = {b0, b1, b2};
        void *ov[3] = {o0, o1, o2};
        int r = WH_ENOSPC;
        trace_begin(TR_DEC_GEMM, s);
        if (g != nullptr)
            r = dec_gemm_launch(mode, nullptr, x, g, b, batch, K, wv, seg_n, N, bv, ov, cap, pos_c, amax, ctl,
                                num_sms, s);
        trace_end(TR_DEC_GEMM, s, 2.0 * batch * (double)N * K,
                  2.0 * (double)N * K + (g != nullptr ? 4.0 : 2.0) * batch * (double)K);
        if (r != WH_ENOSPC) return r;
        if (g != nullptr) {
            trace_begin(TR_DEC_OTHER, s);
            r = layernorm_launch(x, batch, d, g, b, xn, 1, s, true);
            trace_end(TR_DEC_OTHER, s, 0.0, (double)batch * d * 6.0);
            if (r) return r;
            a = xn;
        }
        trace_begin(TR_DEC_GEMM, s);
        r = dec_gemm_launch(mode, a, nullptr, nullptr, nullptr, batch, K, wv, seg_n, N, bv, ov, cap, pos_c, amax, ctl,
                            num_sms, s);
        trace_end(TR_DEC_GEMM, s, 2.0 * batch * (double)N * K, 2.0 * (double)N * K + 2.0 * batch * (double)K);
        return r;
    };
    auto attend = [&](const void *qp, const void *kp, const void *vp, long long row_stride, long long seq_stride,
                      const int *nk, int max_keys, void *da) {
        trace_begin(TR_DEC_ATTN, s);
        const int r = decode_attention_launch(qp, kp, vp, row_stride, seq_stride, nk, max_keys, batch, H, ao, da, ctl,
                                              num_sms, s, true, false);
        trace_end(TR_DEC_ATTN, s, 4.0 * batch * (double)max_keys * d, 4.0 * batch * (double)max_keys * d);
        return r;
    };

    for (int l = 0; l < cfg->n_layer; ++l) {
        const wh_dec_layer_weights &Lw = w->layers[l];
        wh_bf16 *kc = kcache + (size_t)l * layer_cache, *vc = vcache + (size_t)l * layer_cache;
        const wh_bf16 *ckv = cross_kv + (size_t)l * layer_cross;
        // causal self-attention: this token's k / v go to row pos of the caches, then its
        // query attends over rows 0 .. pos
        if ((rc = gemm(SK_QKV, Lw.ln1_g, Lw.ln1_b, xn, d, Lw.wq, Lw.wk, Lw.wv, d, 3 * d, Lw.bq, nullptr, Lw.bv, q, kc,
                       vc)))
            return rc;
        if ((rc = attend(q, kc, vc, d, (long long)cap * d, n_self, cap, da_self))) return rc;
        if ((rc = gemm(SK_RESID, nullptr, nullptr, ao, d, Lw.wo, nullptr, nullptr, d, d, Lw.bo, nullptr, nullptr, x,
                       nullptr, nullptr)))
            return rc;
        // cross-attention into the encoder memory (keys / values cached once per clip)
        if ((rc = gemm(SK_BF16, Lw.lnx_g, Lw.lnx_b, xn, d, Lw.xwq, nullptr, nullptr, d, d, Lw.xbq, nullptr, nullptr, q,
                       nullptr, nullptr)))
            return rc;
        if ((rc = attend(q, ckv, ckv + d, 2LL * d, (long long)n_ctx * 2 * d, nullptr, n_ctx, da_cross))) return rc;
        if ((rc = gemm(SK_RESID, nullptr, nullptr, ao, d, Lw.xwo, nullptr, nullptr, d, d, Lw.xbo, nullptr, nullptr, x,
                       nullptr, nullptr)))
            return rc;
        // feed-forward
        if ((rc = gemm(SK_GELU, Lw.ln2_g, Lw.ln2_b, xn, d, Lw.w1, nullptr, nullptr, f, f, Lw.b1, nullptr, nullptr, hb,
                       nullptr, nullptr)))
            return rc;
        if ((rc = gemm(SK_RESID, nullptr, nullptr, hb, f, Lw.w2, nullptr, nullptr, d, d, Lw.b2, nullptr, nullptr, x,
                       nullptr, nullptr)))
            return rc;
    }
    // final norm, logits through the token embedding, greedy token
    if ((rc = gemm(SK_LOGITS, w->lnf_g, w->lnf_b, xn, d, w->tok_embd, nullptr, nullptr, V, V, nullptr, nullptr,
                   nullptr, logits, nullptr, nullptr)))
        return rc;
    if (next_tok) {
        trace_begin(TR_DEC_OTHER, s);
        rc = dec_argmax_launch(amax, batch, next_tok, s);
        trace_end(TR_DEC_OTHER, s, 0.0, (double)batch * 12.0);
    }
    return rc;
}
