// Dense layers of the encoder on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// C[M][N] = A[M][K] * B[N][K]^T, both operands K-major bf16 (activations [tokens][features]
// and nn.Linear weights [out][in]), fp32 accumulation in TMEM, fused epilogues:
//   QKV projection (bias on q and v only: "whisper 0.9.0 API", model.nu, k_proj has no bias),
//   fc1 + erf-GELU (kernels.nu), out_proj / fc2 + residual add into the fp32 stream,
//   conv1 + GELU written straight into conv2's im2col matrix, conv2 + GELU + stored positions
//   (model.nu: conv1 -> GELU -> conv2 -> GELU, embed_positions added).
//
// Kernel structure (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      one thread issues TMA loads of A/B k-blocks (64 wide, 128-byte swizzle) into
//               a STAGES-deep shared-memory ring (full/empty mbarriers)
//   warp 1      allocates TMEM; one thread issues tcgen05.mma (M=128, N=BN, K=16) into one of
//               two TMEM accumulators and commits stage releases / accumulator-ready barriers
//   warps 2..5  epilogue: tcgen05.ld the accumulator (each warp owns one 32-lane quarter of
//               TMEM = 32 rows), apply bias / GELU / residual / positions, store to global;
//               then release the accumulator so the MMA of tile i+2 can start.
// Every wait is bounded (DevCtl::wait_ns); on expiry the block records WH_ETIMEOUT, winds
// down, waits for its own copies and MMAs in flight, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int GEMM_THREADS = 192;

struct GemmArgs {
    int M, N, num_kb, tiles_n, num_tiles, seg_n;
    const float *bias0, *bias1, *bias2;
    void *out;
    long long ldo;
    const float *pos;
    int rows_per_win;
    DevCtl ctl;
};

struct TmapB {
    CUtensorMap m[3];
};

template <int BN>
struct Cfg {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int TMEM_COLS = 2 * BN;  // two accumulators
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
};

template <int MODE>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs &p, int row, int col, const uint32_t (&r)[32]) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    const int seg = col / p.seg_n;
    const float *bias = seg == 0 ? p.bias0 : (seg == 1 ? p.bias1 : p.bias2);
    if (bias != nullptr) {
        const float4 *b4 = reinterpret_cast<const float4 *>(bias + (col - seg * p.seg_n));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 b = __ldg(b4 + j);
            v[4 * j] += b.x;
            v[4 * j + 1] += b.y;
            v[4 * j + 2] += b.z;
            v[4 * j + 3] += b.w;
        }
    }
    if constexpr (MODE == GEMM_BF16 || MODE == GEMM_GELU_BF16 || MODE == GEMM_CONV1) {
        if constexpr (MODE != GEMM_BF16) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = gelu_erf(v[j]);
        }
        uint4 pk[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            pk[j] = make_uint4(pack_bf16(v[8 * j], v[8 * j + 1]), pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                               pack_bf16(v[8 * j + 4], v[8 * j + 5]), pack_bf16(v[8 * j + 6], v[8 * j + 7]));
        __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.out);
        if constexpr (MODE != GEMM_CONV1) {
            uint4 *dst = reinterpret_cast<uint4 *>(out + (long long)row * p.ldo + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = pk[j];
        } else {
            // Row `row` is conv1 output frame s of window w.  conv2 output t reads frames
            // 2t-1, 2t, 2t+1 as taps 0, 1, 2; its im2col row holds [tap0 | tap1 | tap2] x N.
            const int w = row / p.rows_per_win, s = row - w * p.rows_per_win;
            const int t_out = p.rows_per_win / 2;
            __nv_bfloat16 *base = out + (long long)w * t_out * p.ldo + col;
            auto put = [&](int t, int tap) {
                uint4 *dst = reinterpret_cast<uint4 *>(base + (long long)t * p.ldo + (long long)tap * p.N);
#pragma unroll
                for (int j = 0; j < 4; ++j) dst[j] = pk[j];
            };
            if ((s & 1) == 0) {
                put(s >> 1, 1);
            } else {
                if (((s + 1) >> 1) < t_out) put((s + 1) >> 1, 0);
                put((s - 1) >> 1, 2);
            }
            if (s == 0) {  // output 0, tap 0 reads the zero padding in front of frame 0
                uint4 *dst = reinterpret_cast<uint4 *>(base);
#pragma unroll
                for (int j = 0; j < 4; ++j) dst[j] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    } else if constexpr (MODE == GEMM_RESID_F32) {
        float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + (long long)row * p.ldo + col);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 x = dst[j];
            x.x += v[4 * j];
            x.y += v[4 * j + 1];
            x.z += v[4 * j + 2];
            x.w += v[4 * j + 3];
            dst[j] = x;
        }
    } else {  // GEMM_CONV2
        const float4 *pos4 =
            reinterpret_cast<const float4 *>(p.pos + (long long)(row % p.rows_per_win) * p.N + col);
        float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + (long long)row * p.ldo + col);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 q = __ldg(pos4 + j);
            dst[j] = make_float4(gelu_erf(v[4 * j]) + q.x, gelu_erf(v[4 * j + 1]) + q.y,
                                 gelu_erf(v[4 * j + 2]) + q.z, gelu_erf(v[4 * j + 3]) + q.w);
        }
    }
}

template <int BN, int MODE>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ TmapB tmB, const GemmArgs p) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t *empty = full + C::STAGES;
    uint64_t *tfull = empty + C::STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB.m[0]);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0, issued = 0, last_parity = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
            const int mb = tile / p.tiles_n, nb = tile - mb * p.tiles_n;
            const int n0 = nb * BN, seg = n0 / p.seg_n, nin = n0 - seg * p.seg_n;
            const CUtensorMap *mapB = &tmB.m[seg];
            for (int kb = 0; kb < p.num_kb; ++kb) {
                if (*abort_flag || !mbar_wait(empty + stage, phase ^ 1u, p.ctl)) {
                    ok = false;
                    break;
                }
                uint8_t *sa = smem + stage * C::STAGE_BYTES;
                mbar_arrive_expect_tx(full + stage, C::STAGE_BYTES);
                tma_load_2d(sa, &tmA, full + stage, kb * BK, mb * BM);
                tma_load_2d(sa + C::A_BYTES, mapB, full + stage, kb * BK, nin);
                issued |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) *abort_flag = 1;
        // No copy may still be landing in shared memory when the block exits.
        for (int s = 0; s < C::STAGES; ++s)
            if ((issued >> s) & 1u) mbar_wait(full + s, (last_parity >> s) & 1u, p.ctl);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
            if (*abort_flag || !mbar_wait(tempty + acc, acc_phase ^ 1u, p.ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < p.num_kb; ++kb) {
                if (*abort_flag || !mbar_wait(full + stage, phase, p.ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
                const uint64_t ad = sdesc_sw128(sa), bd = sdesc_sw128(sa + C::A_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16(d_tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), IDESC,
                              (kb | k) != 0 ? 1u : 0u);
                umma_commit(empty + stage);  // frees the stage once these MMAs have read it
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit(tfull + acc);  // accumulator ready for the epilogue
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (!ok) *abort_flag = 1;
        umma_commit(drain);
        mbar_wait(drain, 0, p.ctl);  // every MMA of this block has completed
    } else if (warp >= 2) {
        // ---------------- epilogue ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
            bool ok = !*abort_flag && mbar_wait(tfull + acc, acc_phase, p.ctl);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int mb = tile / p.tiles_n, nb = tile - mb * p.tiles_n;
            const int row = mb * BM + q * 32 + lane;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                tmem_ld32(tbase + (uint32_t)c, r);
                tmem_wait_ld();
                if (row < p.M) epilogue_chunk<MODE>(p, row, nb * BN + c, r);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty + acc);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, int MODE>
int launch_t(const CUtensorMap &ta, const TmapB &tb, const GemmArgs &a, int grid, cudaStream_t s) {
    auto kern = k_gemm<BN, MODE>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<BN>::SMEM_BYTES) !=
        cudaSuccess)
        return WH_ECUDA;
    kern<<<grid, GEMM_THREADS, Cfg<BN>::SMEM_BYTES, s>>>(ta, tb, a);
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

template <int BN>
int launch_mode(int mode, const CUtensorMap &ta, const TmapB &tb, const GemmArgs &a, int grid, cudaStream_t s) {
    switch (mode) {
        case GEMM_BF16: return launch_t<BN, GEMM_BF16>(ta, tb, a, grid, s);
        case GEMM_GELU_BF16: return launch_t<BN, GEMM_GELU_BF16>(ta, tb, a, grid, s);
        case GEMM_RESID_F32: return launch_t<BN, GEMM_RESID_F32>(ta, tb, a, grid, s);
        case GEMM_CONV1: return launch_t<BN, GEMM_CONV1>(ta, tb, a, grid, s);
        case GEMM_CONV2: return launch_t<BN, GEMM_CONV2>(ta, tb, a, grid, s);
    }
    return WH_EINVAL;
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

int tmap_encoder_ready() {
    if (g_encode) return WH_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return WH_ECUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return WH_OK;
}

// 2-D bf16 tensor map over rows x cols (row stride ld elements), box 64 x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
int make_tmap_bf16(CUtensorMap *m, const void *ptr, long long rows, int cols, int ld, int box_rows) {
    if (int rc = tmap_encoder_ready()) return rc;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? WH_OK : WH_EINVAL;
}

int gemm_launch(const GemmDesc &g, int mode, const DevCtl &ctl, int num_sms, cudaStream_t s) {
    if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.seg_n <= 0 || g.N % g.seg_n != 0 || g.N / g.seg_n > 3 ||
        g.seg_n % 128 != 0 || g.K % 8 != 0 || g.lda % 8 != 0 || g.ldb % 8 != 0)
        return WH_EINVAL;
    const int BN = (g.seg_n % 256 == 0) ? 256 : 128;
    const int nseg = g.N / g.seg_n;
    CUtensorMap ta;
    TmapB tb;
    if (int rc = make_tmap_bf16(&ta, g.a, g.M, g.K, g.lda, BM)) return rc;
    for (int i = 0; i < 3; ++i) {
        const void *b = g.b[i < nseg ? i : 0];
        if (int rc = make_tmap_bf16(&tb.m[i], b, g.seg_n, g.K, g.ldb, BN)) return rc;
    }
    GemmArgs a;
    a.M = g.M;
    a.N = g.N;
    a.num_kb = (g.K + BK - 1) / BK;
    a.tiles_n = g.N / BN;
    const int tiles_m = (g.M + BM - 1) / BM;
    a.num_tiles = tiles_m * a.tiles_n;
    a.seg_n = g.seg_n;
    a.bias0 = g.bias[0];
    a.bias1 = nseg > 1 ? g.bias[1] : nullptr;
    a.bias2 = nseg > 2 ? g.bias[2] : nullptr;
    a.out = g.out;
    a.ldo = g.ldo;
    a.pos = g.pos;
    a.rows_per_win = g.rows_per_win;
    a.ctl = ctl;
    const int grid = a.num_tiles < num_sms ? a.num_tiles : num_sms;
    count_launch();
    return BN == 256 ? launch_mode<256>(mode, ta, tb, a, grid, s) : launch_mode<128>(mode, ta, tb, a, grid, s);
}

}  // namespace wh
