// Non-causal multi-head self-attention, head_dim 64, on the 5th-generation tensor cores
// ("whisper 0.9.0 API", kernels.nu: attn_sc scores each query against every key with the
// 1/sqrt(64) scale and no causal mask in the encoder, attn_out weights v by the softmax of
// those scores, attn_f fuses both with an online softmax at head_dim 64;
// "How Audio Becomes Words", section "The Encoder: Understand Once": every frame attends to
// the whole 1500 x 1500 square, no mask, no RoPE).
//
// Work item = two 128-query tiles (t = 0, 1) of one (window, head); keys stream through in
// tiles of 128.  One persistent CTA per SM walks the items (window-major, so CTAs running at
// the same time share K/V in L2); the next item's loads and first Q K^T overlap the current
// item's last steps.  q/k/v are read straight from the QKV projection's output [rows][3 D] by TMA
// (128-byte swizzle).  Per key tile j and query tile t:
//   S_t = Q_t K_j^T            tcgen05.mma M=128 N=128 K=64 into TMEM (128 fp32 columns)
//   softmax warps (4 per tile, one query row per thread) read S_t from TMEM, keep the running
//   row maximum m and sum l, write P = exp2((S - m) / 8 * log2 e) as bf16 pairs into TMEM
//   O_t += P_t V_j             tcgen05.mma M=128 N=64 K=128, A = P from TMEM, V (MN-major)
//                              from shared memory, D in TMEM
//   O_t accumulates in TMEM across key tiles; it is rescaled (by the softmax warps) only when
//   the running maximum grows by more than 2^8 in the exp2 domain
// Each query tile has its own MMA-issuing thread, so one tile's softmax overlaps the other
// tile's MMAs.  Keys at or past n_ctx (the last tile: 1500 = 11 * 128 + 92) are masked; the
// score matrix never leaves the SM.
//
// Roles: warp 0 TMA producer, warp 1 TMEM allocation + MMA issuer of tile 0, warp 2 MMA
// issuer of tile 1 (warp 3 idle), warps 4-7 softmax of tile 0, warps 8-11 softmax of tile 1
// (warp w reads TMEM lanes 32 (w % 4) .. + 31).  Every wait is bounded (DevCtl::wait_ns): on expiry
// the block records WH_ETIMEOUT, winds down, drains its own copies and MMAs, frees TMEM.
#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

constexpr int QT = 128, KT = 128, HD = 64, NST = 4;
constexpr int THREADS = 384;
// Register split (setmaxnreg): launched at 168 per thread (384 x 168 = 64512); the producer /
// MMA warpgroup drops to 88 and the two softmax warpgroups rise to 208:
// 128 x 88 + 256 x 208 = 64512, exactly the launch total.
constexpr int REG_LOW = 88, REG_HIGH = 208;
static_assert(128 * REG_LOW + 256 * REG_HIGH <= THREADS * 168, "register split exceeds the launch total");
constexpr int Q_BYTES = QT * HD * 2;     // 16 KB
constexpr int KV_BYTES = KT * HD * 2;    // 16 KB
constexpr int OFF_Q = 0;
constexpr int OFF_KV = 2 * Q_BYTES;
constexpr int OFF_BAR = OFF_KV + NST * 2 * KV_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
constexpr uint32_t TMEM_COLS = 512;      // S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384)
                                         // P0 [384,448) P1 [448,512) (bf16 pairs)

struct AttnArgs {
    int n_ctx, n_head, nkv;
    int n_qblk, n_items;  // work items: (window, head, block of 2 query tiles), window-major
    __nv_bfloat16 *out;
    float scale_log2;
    DevCtl ctl;
};

__device__ __forceinline__ float ex2(float x) { return ex2_approx(x); }
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// MN-major operand (V: rows = keys (the K dimension), 64 contiguous head dims = one 128-byte
// swizzle atom along N): 8-row K groups 1024 bytes apart.  Only one atom along N, so the
// leading offset is never used; it is set to the same 1024 bytes.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(1024 >> 4) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__global__ void __launch_bounds__(THREADS, 1) k_attention_tc(const __grid_constant__ CUtensorMap tm, const AttnArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sQ = smem + OFF_Q;
    uint8_t *sKV = smem + OFF_KV;      // stage s: K at s * 32 KB, V at s * 32 KB + 16 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *q_full = bars;
    uint64_t *q_empty = q_full + 1;     // both issuers' last Q K^T of an item has completed
    uint64_t *kv_full = q_empty + 1;
    uint64_t *kv_empty = kv_full + NST;
    uint64_t *s_full = kv_empty + NST;
    uint64_t *s_free = s_full + 2;
    uint64_t *p_full = s_free + 2;
    uint64_t *o_full = p_full + 2;
    uint64_t *drain = o_full + 2;
    uint64_t *turn = drain + 2;         // turn[t]: tile t may run its exponentials
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(turn + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.n_head * HD;
    const int nkv = p.nkv;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 2);           // one commit from each MMA issuer
        for (int s = 0; s < NST; ++s) {
            mbar_init(kv_full + s, 1);
            mbar_init(kv_empty + s, 2);  // one commit from each MMA issuer
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(s_full + t, 1);
            mbar_init(s_free + t, 4);
            mbar_init(p_full + t, 4);
            mbar_init(o_full + t, 1);
        }
        mbar_init(drain, 1);
        mbar_init(drain + 1, 1);
        mbar_init(turn, 4);
        mbar_init(turn + 1, 4);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Persistent: this CTA takes items blockIdx.x, blockIdx.x + gridDim.x, ...  Every role walks
    // the same item sequence; K/V tiles and per-tile steps are numbered across items, so the
    // next item's Q and K/V loads and its first Q K^T overlap the end of the current item.
    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_LOW));
      if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        uint32_t issued = 0, last_parity = 0, g = 0;
        int k = 0;
        for (int item = blockIdx.x; item < p.n_items; item += gridDim.x, ++k) {
            const int qb = item % p.n_qblk, bh = item / p.n_qblk;
            const int h = bh % p.n_head, row0 = (bh / p.n_head) * p.n_ctx, q0 = qb * 2 * QT;
            // Q of the previous item is no longer read once both issuers' last Q K^T completed
            if (*abort_flag || (k > 0 && !mbar_wait(q_empty, (uint32_t)(k - 1) & 1u, p.ctl))) {
                *abort_flag = 1;
                break;
            }
            mbar_arrive_expect_tx(q_full, 2 * Q_BYTES);
            tma_load_2d(sQ, &tm, q_full, h * HD, row0 + q0);
            tma_load_2d(sQ + Q_BYTES, &tm, q_full, h * HD, row0 + q0 + QT);
            bool stop = false;
            for (int j = 0; j < nkv; ++j, ++g) {
                const int s = g % NST;
                const uint32_t ph = (g / NST) & 1u;
                if (*abort_flag || !mbar_wait(kv_empty + s, ph ^ 1u, p.ctl)) {
                    *abort_flag = 1;
                    stop = true;
                    break;
                }
                uint8_t *kb = sKV + s * 2 * KV_BYTES;
                mbar_arrive_expect_tx(kv_full + s, 2 * KV_BYTES);
                tma_load_2d(kb, &tm, kv_full + s, D + h * HD, row0 + j * KT);
                tma_load_2d(kb + KV_BYTES, &tm, kv_full + s, 2 * D + h * HD, row0 + j * KT);
                issued |= 1u << s;
                last_parity = (last_parity & ~(1u << s)) | (ph << s);
            }
            if (stop) {
                ++k;  // this item's Q was issued
                break;
            }
        }
        // no copy of this CTA may still be in flight when it exits
        if (k > 0) mbar_wait(q_full, (uint32_t)(k - 1) & 1u, p.ctl);
        for (int s = 0; s < NST; ++s)
            if ((issued >> s) & 1u) mbar_wait(kv_full + s, (last_parity >> s) & 1u, p.ctl);
    } else if ((warp == 1 || warp == 2) && lane == 0) {
        // ---------------- MMA issuers: warp 1 -> query tile 0, warp 2 -> query tile 1 ----------------
        // Per key tile j: S_t(j+1) as soon as the softmax of tile t has read S_t(j), then
        // O_t += P_t(j) V_j once P_t(j) is in TMEM.  One issuing thread per tile keeps a tile's
        // P V from queueing behind the other tile's Q K^T.
        const int t = warp - 1;
        constexpr uint32_t IDESC_S = idesc_bf16_f32(QT, KT);
        constexpr uint32_t IDESC_O = idesc_bf16_f32(QT, HD) | (1u << 16);  // B (V) is MN-major
        const uint32_t sq = smem_u32(sQ) + t * Q_BYTES, skv = smem_u32(sKV);
        const uint32_t dS = tmem + 128u * t, dO = tmem + 256u + 64u * t, aP = tmem + 384u + 64u * t;
        auto issue_s = [&](uint32_t s) {
            const uint64_t a = sdesc_sw128(sq), bk = sdesc_sw128(skv + s * 2 * KV_BYTES);
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk)
                umma_bf16(dS, a + (uint64_t)(2 * kk), bk + (uint64_t)(2 * kk), IDESC_S, kk != 0);
            umma_commit(s_full + t);
        };
        bool ok = true;
        uint32_t g = 0, G = 0;  // K/V tiles consumed, steps of this tile (both across items)
        int k = 0;
        for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x, ++k) {
            // S_t(0) of this item: its Q has landed, K tile 0 has landed, and the softmax has
            // read the previous item's last S_t.
            ok = !*abort_flag && mbar_wait(q_full, (uint32_t)k & 1u, p.ctl) &&
                 mbar_wait(kv_full + g % NST, (g / NST) & 1u, p.ctl) &&
                 (G == 0 || mbar_wait(s_free + t, (G - 1) & 1u, p.ctl));
            if (!ok) break;
            tc_fence_after();
            issue_s(g % NST);
            if (nkv == 1) umma_commit(q_empty);
            for (int j = 0; j < nkv; ++j) {
                const uint32_t s = (g + j) % NST;
                if (j + 1 < nkv) {
                    const uint32_t g1 = g + j + 1;
                    ok = !*abort_flag && mbar_wait(kv_full + g1 % NST, (g1 / NST) & 1u, p.ctl) &&
                         mbar_wait(s_free + t, (G + j) & 1u, p.ctl);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(g1 % NST);
                    if (j + 2 == nkv) umma_commit(q_empty);  // the item's last Q K^T
                }
                ok = !*abort_flag && mbar_wait(p_full + t, (G + j) & 1u, p.ctl);
                if (!ok) break;
                tc_fence_after();
                const uint32_t vb = skv + s * 2 * KV_BYTES + KV_BYTES;
#pragma unroll
                for (int kk = 0; kk < KT / 16; ++kk)  // P (A operand) from TMEM: 16 keys = 8 columns
                    umma_bf16_tmem_a(dO, aP + 8u * kk, sdesc_sw128_mn(vb + kk * 2048), IDESC_O, (j | kk) != 0);
                umma_commit(o_full + t);
                umma_commit(kv_empty + s);  // one of the two arrivals that free K/V stage s
            }
            g += nkv;
            G += nkv;
        }
        if (!ok) *abort_flag = 1;
        umma_commit(drain + t);
        mbar_wait(drain + t, 0, p.ctl);
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REG_HIGH));
        // ---------------- softmax: one query row per thread ----------------
        // O accumulates in TMEM.  The row maximum m used for the exponentials is only raised
        // (and O, l rescaled) when the true maximum exceeds it by more than 2^8 in the exp2
        // domain, so exponentials stay <= 256 and the rescale is rare.
        const int t = (warp - 4) >> 2;
        const int r = (warp & 3) * 32 + lane;                 // TMEM lane quarter = warp % 4
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + 128u * t;
        const uint32_t tO = tmem + lane_off + 256u + 64u * t;
        const uint32_t tP = tmem + lane_off + 384u + 64u * t;
        const float sl2 = p.scale_log2;
        bool ok = true;
        uint32_t G = 0;                                        // steps of this tile across items
        if (t == 1 && lane == 0) mbar_arrive(turn);            // tile 0 takes the first turn
        for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
            const int qb = item % p.n_qblk, bh = item / p.n_qblk;
            const int h = bh % p.n_head, row0 = (bh / p.n_head) * p.n_ctx, q0 = qb * 2 * QT;
            const bool last_item = item + (int)gridDim.x >= p.n_items;
            float m = -INFINITY, l = 0.0f;
            for (int j = 0; j < nkv; ++j) {
                const uint32_t par = (G + j) & 1u;
                ok = __all_sync(0xffffffffu, !*abort_flag && mbar_wait(s_full + t, par, p.ctl));
                if (!ok) break;
                tc_fence_after();
                uint32_t sv[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32u * c, sv[c]);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free + t);           // S_t may now be overwritten
                const int kvalid = p.n_ctx - j * KT;               // keys of this tile inside the window
                if (kvalid < KT) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (32 * c + i >= kvalid) sv[c][i] = 0xff800000u;  // -inf
                }
                // row maximum: 8 independent partial maxima, then a tree (no 128-long chain)
                float pm[8];
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) pm[kk] = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; i += 2)
                        pm[(i >> 1) & 7] = max3(pm[(i >> 1) & 7], __uint_as_float(sv[c][i]), __uint_as_float(sv[c][i + 1]));
                const float mx = max3(max3(pm[0], pm[1], pm[2]), max3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
                const float m_new = fmaxf(m, mx);
                if (j == 0) {
                    m = m_new;
                } else {
                    // PV of the previous tile is done: O is stable and the P buffer is free.
                    ok = __all_sync(0xffffffffu, mbar_wait(o_full + t, par ^ 1u, p.ctl));
                    if (!ok) break;
                    tc_fence_after();
                    const bool need = (m_new - m) * sl2 > 8.0f;
                    if (__any_sync(0xffffffffu, need)) {
                        float f = 1.0f;
                        if (need) {
                            f = ex2((m - m_new) * sl2);
                            l *= f;
                            m = m_new;
                        }
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t v[32];
                            tmem_ld32(tO + 32u * half, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                            tmem_st32(tO + 32u * half, v);
                        }
                        tmem_wait_st();
                    }
                }
                // Scale and subtract the maximum (packed fp32, two keys per instruction) before
                // this tile's turn, so the turn holds only the exponentials and the P store.
                const float mc = m * sl2;
                const uint64_t sl2x2 = f2_pack(sl2, sl2), nmcx2 = f2_pack(-mc, -mc);
                uint64_t xv[64];                                   // key pairs 2k, 2k + 1
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; i += 2)
                        xv[16 * c + (i >> 1)] =
                            fma_f2(f2_pack(__uint_as_float(sv[c][i]), __uint_as_float(sv[c][i + 1])), sl2x2, nmcx2);
                // Ping-pong: the two tiles take turns in the exponential section, so one tile's
                // S load, row maximum, scaling, row sum and waits overlap the other tile's
                // exponentials.
                ok = __all_sync(0xffffffffu, mbar_wait(turn + t, par, p.ctl));
                if (!ok) break;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {                   // 64 keys -> 32 packed bf16 pairs
                    uint32_t pk[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        float x0, x1;
                        f2_unpack(xv[32 * hh + k], x0, x1);
                        const float e0 = ex2(x0), e1 = ex2(x1);
                        xv[32 * hh + k] = f2_pack(e0, e1);
                        pk[k] = pack_bf16(e0, e1);
                    }
                    tmem_st32(tP + 32u * hh, pk);
                }
                __syncwarp();
                // tile 1's very last step is the CTA's last turn
                if (lane == 0 && (t == 0 || !(last_item && j + 1 == nkv))) mbar_arrive(turn + (1 - t));
                {
                    // row sum of the exponentials: 4 x 2 independent partial sums, keys in order
                    uint64_t ps[4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) ps[kk] = 0ull;
#pragma unroll
                    for (int k = 0; k < 64; ++k) ps[k & 3] = add_f2(ps[k & 3], xv[k]);
                    const uint64_t s2 = add_f2(add_f2(ps[0], ps[1]), add_f2(ps[2], ps[3]));
                    float a0, a1;
                    f2_unpack(s2, a0, a1);
                    l += a0 + a1;
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full + t);
            }
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_full + t, (G + nkv - 1) & 1u, p.ctl));
            if (!ok) break;
            tc_fence_after();
            const float inv = 1.0f / l;
            const int q = q0 + t * QT + r;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t v[32];
                tmem_ld32(tO + 32u * half, v);
                tmem_wait_ld();
                if (q < p.n_ctx) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((long long)row0 + q) * D + h * HD + 32 * half);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t w[4];
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            w[kk] = pack_bf16(__uint_as_float(v[8 * c + 2 * kk]) * inv,
                                              __uint_as_float(v[8 * c + 2 * kk + 1]) * inv);
                        dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            // O has been read: the next item's first P V may overwrite it (its p_full follows)
            tc_fence_before();
            G += nkv;
        }
        if (!ok) *abort_flag = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

int attention_prepare() {
    return cudaFuncSetAttribute(k_attention_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) == cudaSuccess
               ? WH_OK
               : WH_ECUDA;
}

int attention_launch(const void *qkv, int batch, int n_ctx, int n_head, void *out, const DevCtl &ctl,
                     int num_sms, cudaStream_t s) {
    if (batch <= 0) return WH_OK;
    const int D = n_head * HD;
    CUtensorMap tm;
    if (int rc = make_tmap_bf16(&tm, qkv, (long long)batch * n_ctx, 3 * D, 3 * D, 128)) return rc;
    AttnArgs a;
    a.n_ctx = n_ctx;
    a.n_head = n_head;
    a.nkv = (n_ctx + KT - 1) / KT;
    a.n_qblk = (n_ctx + 2 * QT - 1) / (2 * QT);
    const long long items = (long long)a.n_qblk * n_head * batch;
    if (items > (1LL << 30)) return WH_EINVAL;
    a.n_items = (int)items;
    a.out = reinterpret_cast<__nv_bfloat16 *>(out);
    a.scale_log2 = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)
    a.ctl = ctl;
    // one CTA per SM (shared memory and TMEM allow no second), persistent over the items
    const int grid = a.n_items < num_sms ? a.n_items : num_sms;
    k_attention_tc<<<grid, THREADS, SMEM_BYTES, s>>>(tm, a);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

}  // namespace wh
