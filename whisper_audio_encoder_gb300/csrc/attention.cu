// Non-causal multi-head self-attention, head_dim 64 ("whisper 0.9.0 API", kernels.nu:
// attn_f "fused attention, online softmax (hd = 64)", attn_sc "scores = q.k / sqrt(hd), NO
// causal mask", attn_out "softmax(scores) . v"; "How Audio Becomes Words", section "The
// Encoder: Understand Once": the full 1500 x 1500 square, no mask, no RoPE).
//
// Flash-style: one block = 64 queries of one (window, head), 4 warps x 16 query rows.
// K/V tiles of 64 keys stream through a double-buffered shared-memory ring (cp.async,
// XOR-swizzled 16-byte chunks); S = Q K^T and O += P V on bf16 tensor-core MMAs with fp32
// accumulation; the softmax is online in registers (running max and sum per row, base-2
// exponent with the 1/8 * log2(e) scale folded in).  Keys past n_ctx (the 1500 = 23 * 64 + 28
// tail) are masked with -inf; the score matrix never reaches memory.
#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

constexpr int BQ = 64, BKV = 64, ATT_THREADS = 128;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Byte offset of 16-byte chunk `ch` of row `r` in a [64][64] bf16 tile (128-byte rows).
__device__ __forceinline__ uint32_t toff(int r, int ch) { return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4)); }

__global__ void __launch_bounds__(ATT_THREADS) k_attention(const __nv_bfloat16 *__restrict__ qkv, int n_ctx,
                                                           int n_head, __nv_bfloat16 *__restrict__ out,
                                                           float scale_log2) {
    __shared__ __align__(128) uint8_t sQ[BQ * 128];
    __shared__ __align__(128) uint8_t sK[2][BKV * 128];
    __shared__ __align__(128) uint8_t sV[2][BKV * 128];
    const int h = blockIdx.y, b = blockIdx.z;
    const int D = n_head * 64;
    const long long ld = 3LL * D;
    const __nv_bfloat16 *base = qkv + (long long)b * n_ctx * ld;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q0 = blockIdx.x * BQ;

    for (int c = tid; c < BQ * 8; c += ATT_THREADS) {
        const int r = c >> 3, ch = c & 7, qr = q0 + r;
        const __nv_bfloat16 *src = base + (long long)min(qr, n_ctx - 1) * ld + h * 64 + ch * 8;
        cp_async16(smem_u32(sQ) + toff(r, ch), src, qr < n_ctx ? 16 : 0);
    }
    auto load_kv = [&](int j, int buf) {
        const int k0 = j * BKV;
        for (int c = tid; c < BKV * 8; c += ATT_THREADS) {
            const int r = c >> 3, ch = c & 7, kr = k0 + r;
            const long long roff = (long long)min(kr, n_ctx - 1) * ld + h * 64 + ch * 8;
            const int bytes = kr < n_ctx ? 16 : 0;
            cp_async16(smem_u32(sK[buf]) + toff(r, ch), base + roff + D, bytes);
            cp_async16(smem_u32(sV[buf]) + toff(r, ch), base + roff + 2 * D, bytes);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    const int nkv = (n_ctx + BKV - 1) / BKV;
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    uint32_t qf[4][4];
    const int mi = lane >> 3, r8 = lane & 7;

    for (int j = 0; j < nkv; ++j) {
        const int buf = j & 1;
        if (j + 1 < nkv) load_kv(j + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait1();
        __syncthreads();
        if (j == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                ldsm_x4(smem_u32(sQ) + toff(warp * 16 + (mi & 1) * 8 + r8, kk * 2 + (mi >> 1)), qf[kk][0], qf[kk][1],
                        qf[kk][2], qf[kk][3]);
        }
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.0f;
        const uint32_t kbase = smem_u32(sK[buf]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + toff((2 * np + (mi >> 1)) * 8 + r8, kk * 2 + (mi & 1)), b0, b1, b2, b3);
                mma16816(s[2 * np], qf[kk], b0, b1);
                mma16816(s[2 * np + 1], qf[kk], b2, b3);
            }
        const bool tail = (j + 1) * BKV > n_ctx;
        float mx0 = m0, mx1 = m1;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v = s[nt][e] * scale_log2;
                if (tail && j * BKV + nt * 8 + (lane & 3) * 2 + (e & 1) >= n_ctx) v = -INFINITY;
                s[nt][e] = v;
            }
            mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float a0 = ex2(m0 - mx0), a1 = ex2(m1 - mx1);
        m0 = mx0;
        m1 = mx1;
        float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            s[nt][0] = ex2(s[nt][0] - m0);
            s[nt][1] = ex2(s[nt][1] - m0);
            s[nt][2] = ex2(s[nt][2] - m1);
            s[nt][3] = ex2(s[nt][3] - m1);
            rs0 += s[nt][0] + s[nt][1];
            rs1 += s[nt][2] + s[nt][3];
            o[nt][0] *= a0;
            o[nt][1] *= a0;
            o[nt][2] *= a1;
            o[nt][3] *= a1;
        }
        l0 = l0 * a0 + rs0;
        l1 = l1 * a1 + rs1;
        uint32_t pf[4][4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            pf[kk][0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
            pf[kk][1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
            pf[kk][2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pf[kk][3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
        }
        const uint32_t vbase = smem_u32(sV[buf]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + toff(kk * 16 + (mi & 1) * 8 + r8, 2 * np + (mi >> 1)), b0, b1, b2, b3);
                mma16816(o[2 * np], pf[kk], b0, b1);
                mma16816(o[2 * np + 1], pf[kk], b2, b3);
            }
        __syncthreads();
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = 1.0f / l0, i1 = 1.0f / l1;
    const int r0 = q0 + warp * 16 + (lane >> 2), r1 = r0 + 8;
    uint32_t *o0 = reinterpret_cast<uint32_t *>(out + ((long long)b * n_ctx + r0) * D + h * 64);
    uint32_t *o1 = reinterpret_cast<uint32_t *>(out + ((long long)b * n_ctx + r1) * D + h * 64);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        const int c2 = nt * 4 + (lane & 3);  // bf16 pair index within the head
        if (r0 < n_ctx) o0[c2] = pack_bf16(o[nt][0] * i0, o[nt][1] * i0);
        if (r1 < n_ctx) o1[c2] = pack_bf16(o[nt][2] * i1, o[nt][3] * i1);
    }
}

}  // namespace

int attention_launch(const void *qkv, int batch, int n_ctx, int n_head, void *out, cudaStream_t s) {
    if (batch <= 0) return WH_OK;
    dim3 grid((n_ctx + BQ - 1) / BQ, n_head, batch);
    const float scale_log2 = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)
    k_attention<<<grid, ATT_THREADS, 0, s>>>(reinterpret_cast<const __nv_bfloat16 *>(qkv), n_ctx, n_head,
                                             reinterpret_cast<__nv_bfloat16 *>(out), scale_log2);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

}  // namespace wh
