// LayerNorm ("whisper 0.9.0 API", kernels.nu: LayerNorm, not RMSNorm -- it subtracts the
// mean and it has a bias): y = (x - mean) / sqrt(var + 1e-5) * g + b, biased variance.
// One warp per row, the row held in registers (d <= 2048: <= 16 float4 per lane), two
// passes over the registers (mean, then centred variance), warp-shuffle reductions.
// HBM-bound: reads 4 d bytes and writes 2 d (bf16) or 4 d (fp32) bytes per row.
#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

constexpr int LN_THREADS = 256;
constexpr int MAXV = 16;  // float4 per lane: d <= 2048

// d a multiple of 128: each lane holds d / 128 float4 (16-byte loads and stores).  NV > 0
// fixes d = 128 NV at compile time (registers sized to the row: more rows in flight per SM);
// NV = 0 takes d at run time (up to MAXV float4 per lane).
// reverse: blocks take the rows from the last one down (the rows a GEMM stored last are the ones
// still in L2).
template <int NV, bool OUT_BF16>
__global__ void __launch_bounds__(LN_THREADS) k_layernorm(const float *__restrict__ x, int rows, int d,
                                                          const float *__restrict__ g,
                                                          const float *__restrict__ b, void *__restrict__ y,
                                                          int reverse) {
    constexpr int CAP = NV > 0 ? NV : MAXV;
    int row = blockIdx.x * (LN_THREADS / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();
    if (row >= rows) return;
    if (reverse) row = rows - 1 - row;
    const int nv = NV > 0 ? NV : d >> 7;
    if (NV > 0) d = NV * 128;
    const float4 *xr = reinterpret_cast<const float4 *>(x + (long long)row * d);
    float4 v[CAP];
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int i = 0; i < CAP; ++i)
        if (i < nv) v[i] = __ldg(xr + i * 32 + lane);
#pragma unroll
    for (int i = 0; i < CAP; ++i)
        if (i < nv) {
            s0 += v[i].x + v[i].y;
            s1 += v[i].z + v[i].w;
        }
    const float mean = warp_sum(s0 + s1) / (float)d;
    float q0 = 0.0f, q1 = 0.0f;
#pragma unroll
    for (int i = 0; i < CAP; ++i)
        if (i < nv) {
            const float a = v[i].x - mean, bb = v[i].y - mean, c = v[i].z - mean, e = v[i].w - mean;
            q0 = fmaf(a, a, fmaf(bb, bb, q0));
            q1 = fmaf(c, c, fmaf(e, e, q1));
        }
    const float rstd = 1.0f / sqrtf(warp_sum(q0 + q1) / (float)d + 1e-5f);
    const float4 *g4 = reinterpret_cast<const float4 *>(g);
    const float4 *b4 = reinterpret_cast<const float4 *>(b);
#pragma unroll
    for (int i = 0; i < CAP; ++i)
        if (i < nv) {
            const int c = i * 32 + lane;
            const float4 gg = __ldg(g4 + c), bb = __ldg(b4 + c);
            const float o0 = (v[i].x - mean) * rstd * gg.x + bb.x;
            const float o1 = (v[i].y - mean) * rstd * gg.y + bb.y;
            const float o2 = (v[i].z - mean) * rstd * gg.z + bb.z;
            const float o3 = (v[i].w - mean) * rstd * gg.w + bb.w;
            if constexpr (OUT_BF16) {
                reinterpret_cast<uint2 *>(y)[(long long)row * (d >> 2) + c] = make_uint2(pack_bf16(o0, o1), pack_bf16(o2, o3));
            } else {
                reinterpret_cast<float4 *>(y)[(long long)row * (d >> 2) + c] = make_float4(o0, o1, o2, o3);
            }
        }
}

// Launch configuration; with pdl the kernel may start while the previous kernel of the stream
// is still running (it waits for that kernel's results before reading x).
cudaLaunchConfig_t ln_config(int grid, cudaStream_t s, bool pdl, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(LN_THREADS);
    lc.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = pdl ? 1 : 0;
    return lc;
}

template <int NV>
cudaError_t launch_ln(int grid, cudaStream_t s, bool pdl, const float *x, int rows, int d, const float *g,
                      const float *b, void *y, int y_bf16, int rev) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t lc = ln_config(grid, s, pdl, attr);
    return y_bf16 ? cudaLaunchKernelEx(&lc, k_layernorm<NV, true>, x, rows, d, g, b, y, rev)
                  : cudaLaunchKernelEx(&lc, k_layernorm<NV, false>, x, rows, d, g, b, y, rev);
}

// d a multiple of 64 but not of 128: float2 per lane.
template <bool OUT_BF16>
__global__ void __launch_bounds__(LN_THREADS) k_layernorm64(const float *__restrict__ x, int rows, int d,
                                                            const float *__restrict__ g,
                                                            const float *__restrict__ b, void *__restrict__ y,
                                                            int reverse) {
    int row = blockIdx.x * (LN_THREADS / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();
    if (row >= rows) return;
    if (reverse) row = rows - 1 - row;
    const int nv = d >> 6;
    const float2 *xr = reinterpret_cast<const float2 *>(x + (long long)row * d);
    float2 v[2 * MAXV];
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 2 * MAXV; ++i)
        if (i < nv) {
            v[i] = __ldg(xr + i * 32 + lane);
            s += v[i].x + v[i].y;
        }
    const float mean = warp_sum(s) / (float)d;
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < 2 * MAXV; ++i)
        if (i < nv) {
            const float dx = v[i].x - mean, dy = v[i].y - mean;
            q = fmaf(dx, dx, fmaf(dy, dy, q));
        }
    const float rstd = 1.0f / sqrtf(warp_sum(q) / (float)d + 1e-5f);
    const float2 *g2 = reinterpret_cast<const float2 *>(g);
    const float2 *b2 = reinterpret_cast<const float2 *>(b);
#pragma unroll
    for (int i = 0; i < 2 * MAXV; ++i)
        if (i < nv) {
            const int c = i * 32 + lane;
            const float2 gg = __ldg(g2 + c), bb = __ldg(b2 + c);
            const float o0 = (v[i].x - mean) * rstd * gg.x + bb.x;
            const float o1 = (v[i].y - mean) * rstd * gg.y + bb.y;
            if constexpr (OUT_BF16) {
                reinterpret_cast<uint32_t *>(y)[(long long)row * (d >> 1) + c] = pack_bf16(o0, o1);
            } else {
                reinterpret_cast<float2 *>(y)[(long long)row * (d >> 1) + c] = make_float2(o0, o1);
            }
        }
}

}  // namespace

int layernorm_launch(const float *x, int rows, int d, const float *g, const float *b, void *y, int y_bf16,
                     cudaStream_t s, bool pdl, bool reverse) {
    const int rev = reverse ? 1 : 0;
    if (rows <= 0) return WH_OK;
    if (d % 64 != 0 || d < 64 || d > 128 * MAXV) return WH_EINVAL;
    const int grid = (rows + LN_THREADS / 32 - 1) / (LN_THREADS / 32);
    cudaError_t e;
    if (d % 128 == 0) {
        switch (d / 128) {  // the family's widths (384, 512, 768, 1024, 1280) get exact registers
            case 3: e = launch_ln<3>(grid, s, pdl, x, rows, d, g, b, y, y_bf16, rev); break;
            case 4: e = launch_ln<4>(grid, s, pdl, x, rows, d, g, b, y, y_bf16, rev); break;
            case 6: e = launch_ln<6>(grid, s, pdl, x, rows, d, g, b, y, y_bf16, rev); break;
            case 8: e = launch_ln<8>(grid, s, pdl, x, rows, d, g, b, y, y_bf16, rev); break;
            case 10: e = launch_ln<10>(grid, s, pdl, x, rows, d, g, b, y, y_bf16, rev); break;
            default: e = launch_ln<0>(grid, s, pdl, x, rows, d, g, b, y, y_bf16, rev); break;
        }
    } else {
        cudaLaunchAttribute attr[1];
        const cudaLaunchConfig_t lc = ln_config(grid, s, pdl, attr);
        e = y_bf16 ? cudaLaunchKernelEx(&lc, k_layernorm64<true>, x, rows, d, g, b, y, rev)
                   : cudaLaunchKernelEx(&lc, k_layernorm64<false>, x, rows, d, g, b, y, rev);
    }
    count_launch();
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

}  // namespace wh
