// Dense layers of the encoder on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// C[M][N] = A[M][K] * B[N][K]^T, both operands K-major bf16 (activations [tokens][features]
// and nn.Linear weights [out][in]), fp32 accumulation in TMEM, fused epilogues:
//   QKV projection (bias on q and v only: "whisper 0.9.0 API", model.nu, k_proj has no bias),
//   fc1 + erf-GELU (kernels.nu), out_proj / fc2 + residual add into the fp32 stream,
//   conv1 + GELU written straight into conv2's im2col matrix, conv2 + GELU + stored positions
//   (model.nu: conv1 -> GELU -> conv2 -> GELU, embed_positions added).
//
// Kernel structure: persistent CTA pairs (a cluster of two CTAs on two SMs, cta_group::2),
// each pair walking 256 x BN output tiles (BN = 256, or 128 when a segment is not a multiple
// of 256), k-blocks 64 wide:
//   warp 0      (both CTAs) one thread issues TMA loads of this CTA's 128 rows of A and BN/2
//               rows of B (128-byte swizzle) into a STAGES-deep shared-memory ring
//   warp 1      allocates TMEM in both CTAs; on the even CTA one thread issues tcgen05.mma
//               (M=256, N=BN, K=16) reading both CTAs' operand halves, into one of two TMEM
//               accumulators, and multicasts its commits to both CTAs
//   warps 2..9  (both CTAs) epilogue on this CTA's 128 rows: tcgen05.ld, bias / GELU /
//               residual / positions, TMA store through a per-warp staging tile; then hand
//               the accumulator back so the MMA of tile i+2 can start.
// Tiles go to the pairs round-robin.  A long-K residual GEMM whose tiles do not fill whole
// rounds shares the k-blocks of its last rounds evenly between the pairs instead (stream-K,
// see GemmArgs::sk); a tile cut between two pairs is summed in two pieces and merged by the
// second to finish, without waiting.
// Every wait is bounded (DevCtl::wait_ns); on expiry the block records WH_ETIMEOUT, winds
// down, waits for its own copies and MMAs in flight, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

constexpr int BK = 64;
constexpr int GEMM_THREADS = 320;  // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int EPI_WARPS = 8;
constexpr int GEMM_SK_MIN_KB = 64;   // stream-K only for k-loops of at least this many k-blocks

struct GemmArgs {
    int M, N, num_kb, tiles_n, num_tiles, seg_n;
    const float *bias0, *bias1, *bias2;
    void *out;
    long long ldo;
    const float *pos;
    int rows_per_win;
    // Stream-K (residual mode): the first sk_first tiles go round-robin in whole rounds; the
    // W = (num_tiles - sk_first) * num_kb k-blocks of the rest are shared out in tile order,
    // pair p of P taking [p W / P, (p + 1) W / P), so every pair gets the same work.  A tile
    // cut by a pair boundary b is summed by pairs b - 1 (its lower k-blocks, at the end of that
    // pair's share) and b (its upper k-blocks, first in its share); both write their fp32
    // partial to slot b of the workspace (tmB.w), and the second to arrive (an atomic ticket
    // per slot, CTA and epilogue warp; nothing waits) adds the two, the bias and the residual.
    int sk, sk_first;
    long long sk_total;
    int *sk_tickets;  // [slot][CTA of the pair][epilogue warp], zero between launches
    DevCtl ctl;
};

struct TmapB {
    CUtensorMap m[3];
    CUtensorMap w;  // stream-K partials: fp32 [slot][2 parts][256 rows][BN], 32 x 32 boxes
};

// The k-block segments one CTA pair computes, in order: whole tiles pair, pair + P, ... or,
// with stream-K, the tile pieces of its share.  Producer, MMA issuer and epilogue walk the same
// sequence.
struct Walk {
    long long g, g1;
    int next_tile, npairs, sk, rr_end;
    __device__ __forceinline__ Walk(const GemmArgs &p, int pair, int np) : npairs(np), sk(p.sk) {
        next_tile = pair;
        rr_end = sk ? p.sk_first : p.num_tiles;
        const long long base = (long long)p.sk_first * p.num_kb;
        g = sk ? base + (long long)pair * p.sk_total / np : 0;
        g1 = sk ? base + (long long)(pair + 1) * p.sk_total / np : 0;
    }
    __device__ __forceinline__ bool next(const GemmArgs &p, int &tile, int &kb0, int &kb1) {
        if (next_tile < rr_end) {
            tile = next_tile;
            kb0 = 0;
            kb1 = p.num_kb;
            next_tile += npairs;
            return true;
        }
        if (sk) {
            if (g >= g1) return false;
            tile = (int)(g / p.num_kb);
            const long long t0 = (long long)tile * p.num_kb;
            const long long end = g1 < t0 + p.num_kb ? g1 : t0 + p.num_kb;
            kb0 = (int)(g - t0);
            kb1 = (int)(end - t0);
            g = end;
            return true;
        }
        return false;
    }
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

// ---------------------------------------------------------------------------------------
// CTA-pair version (cta_group::2): a cluster of two CTAs computes a 256 x BN tile.  Each
// CTA stages its own 128 rows of A and BN/2 rows of B per k-block; the even CTA issues one
// tcgen05.mma with M = 256 that reads the A and B halves from both CTAs' shared memory, and
// each CTA's TMEM receives its own 128 rows of the accumulator.  Per tensor-core cycle each
// SM now brings in 2/3 of the operand bytes of the single-CTA 128 x 256 tile.
//   full[s]    (even CTA) TMA bytes of both CTAs + the even producer's expect_tx arrival
//   empty[s]   (both)     the even CTA's commit, multicast to both CTAs
//   tfull[a]   (both)     the even CTA's commit, multicast to both CTAs
//   tempty[a]  (even CTA) 4 epilogue warps of each CTA (8 arrivals)
// ---------------------------------------------------------------------------------------
template <int BN>
struct Cfg2 {
    static constexpr int A_BYTES = 128 * BK * 2;
    static constexpr int B_BYTES = (BN / 2) * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = BN == 256 ? 5 : 6;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int EPI_BUF = 8192;  // per epilogue warp: 32 rows x 64 fp32 / bf16 columns
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = EPI_OFF + EPI_WARPS * EPI_BUF;
    static constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory per block");
    static_assert((2 * STAGES + 5 + EPI_WARPS) * 8 + 8 <= 256, "barrier area");
};

// Bias (per output segment) and, for GELU modes, the activation, on 32 accumulator columns.
template <int MODE>
__device__ __forceinline__ void bias_act(const GemmArgs &p, int col, const uint32_t (&r)[32], float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    const int seg = col / p.seg_n;
    const float *bias = seg == 0 ? p.bias0 : (seg == 1 ? p.bias1 : p.bias2);
    if (bias != nullptr) {
        const float4 *b4 = reinterpret_cast<const float4 *>(bias + (col - seg * p.seg_n));
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // packed pairs
            const float4 b = __ldg(b4 + j);
            f2_unpack(add_f2(f2_pack(v[4 * j], v[4 * j + 1]), f2_pack(b.x, b.y)), v[4 * j], v[4 * j + 1]);
            f2_unpack(add_f2(f2_pack(v[4 * j + 2], v[4 * j + 3]), f2_pack(b.z, b.w)), v[4 * j + 2], v[4 * j + 3]);
        }
    }
    if constexpr (MODE == GEMM_GELU_BF16) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) gelu_erf2(v[j], v[j + 1]);
    }
}

// Orders this thread's completed bulk-async (TMA) global accesses with its later generic
// ones, and the other way round.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Epilogue of a stream-K piece of a tile (residual mode), for this warp's 32 rows x BN / 2
// columns.  The raw fp32 sum over the piece's k-blocks goes to its half of the slot through
// the staging tile; once those stores are complete the warp takes the ticket.  The first warp
// to arrive hands its accumulator back and is done.  The second adds the other half's partial
// (a + b: the same bits whichever half is its own), then the bias, into the residual stream.
// Returns false if a wait ran out.
template <int BN>
__device__ __forceinline__ bool sk_epilogue(const GemmArgs &p, const CUtensorMap *tmW, const CUtensorMap *tmOut,
                                            uint8_t *ebuf, uint64_t *xb, uint32_t &xphase, uint32_t tbase,
                                            uint32_t tempty_remote, int slot, int part, int wrow_base, int row0,
                                            int colw, int col, int *ticket, int lane) {
    const int sw = lane & 7;
    uint8_t *mine = ebuf + lane * 128;
    const int wrow = wrow_base + part * 256, orow = wrow_base + (1 - part) * 256;
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += 64) {
        if (lane == 0) bulk_wait_read0();  // the previous store has finished reading ebuf
        __syncwarp();
        uint32_t r0[32], r1[32];
        tmem_ld32(tbase + (uint32_t)c, r0);
        tmem_ld32(tbase + (uint32_t)c + 32u, r1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            *reinterpret_cast<uint4 *>(mine + ((j ^ sw) << 4)) = make_uint4(r0[4 * j], r0[4 * j + 1], r0[4 * j + 2], r0[4 * j + 3]);
            *reinterpret_cast<uint4 *>(mine + 4096 + ((j ^ sw) << 4)) =
                make_uint4(r1[4 * j], r1[4 * j + 1], r1[4 * j + 2], r1[4 * j + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmW, ebuf, colw + c, wrow);
            tma_store_2d(tmW, ebuf + 4096, colw + c + 32, wrow);
            bulk_commit();
        }
    }
    int t = 0;
    if (lane == 0) {
        bulk_wait0();  // this half's partial is in global memory
        fence_proxy_async_global();
        __threadfence();
        t = atomicAdd(ticket, 1);
    }
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t == 0) {  // the other half will finish the tile
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_remote);
        return true;
    }
    if (lane == 0) {
        *ticket = 0;  // both halves have arrived: ready for the next launch
        __threadfence();
        fence_proxy_async_global();
    }
    __syncwarp();
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += 64) {
        if (lane == 0) {
            bulk_wait_read0();
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(xb, 2 * 4096);
            tma_load_2d(ebuf, tmW, xb, colw + c, orow);
            tma_load_2d(ebuf + 4096, tmW, xb, colw + c + 32, orow);
        }
        __syncwarp();
        uint32_t r0[32], r1[32];
        tmem_ld32(tbase + (uint32_t)c, r0);
        tmem_ld32(tbase + (uint32_t)c + 32u, r1);
        tmem_wait_ld();
        if (c + 64 >= BN / 2) {  // last TMEM read of this piece: hand the accumulator back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_remote);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(xb, xphase, p.ctl))) return false;
        xphase ^= 1u;
        float v0[32], v1[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 a = *reinterpret_cast<const float4 *>(mine + ((j ^ sw) << 4));
            const float4 b = *reinterpret_cast<const float4 *>(mine + 4096 + ((j ^ sw) << 4));
            v0[4 * j] = __uint_as_float(r0[4 * j]) + a.x;
            v0[4 * j + 1] = __uint_as_float(r0[4 * j + 1]) + a.y;
            v0[4 * j + 2] = __uint_as_float(r0[4 * j + 2]) + a.z;
            v0[4 * j + 3] = __uint_as_float(r0[4 * j + 3]) + a.w;
            v1[4 * j] = __uint_as_float(r1[4 * j]) + b.x;
            v1[4 * j + 1] = __uint_as_float(r1[4 * j + 1]) + b.y;
            v1[4 * j + 2] = __uint_as_float(r1[4 * j + 2]) + b.z;
            v1[4 * j + 3] = __uint_as_float(r1[4 * j + 3]) + b.w;
        }
        if (p.bias0 != nullptr) {
            const float4 *b0 = reinterpret_cast<const float4 *>(p.bias0 + col + c);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 ba = __ldg(b0 + j), bb = __ldg(b0 + 8 + j);
                v0[4 * j] += ba.x; v0[4 * j + 1] += ba.y; v0[4 * j + 2] += ba.z; v0[4 * j + 3] += ba.w;
                v1[4 * j] += bb.x; v1[4 * j + 1] += bb.y; v1[4 * j + 2] += bb.z; v1[4 * j + 3] += bb.w;
            }
        }
        fence_proxy_async_smem();  // every lane has read the partial before the residual tile replaces it
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_expect_tx(xb, 2 * 4096);
            tma_load_2d(ebuf, tmOut, xb, col + c, row0);
            tma_load_2d(ebuf + 4096, tmOut, xb, col + c + 32, row0);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(xb, xphase, p.ctl))) return false;
        xphase ^= 1u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 *a = reinterpret_cast<float4 *>(mine + ((j ^ sw) << 4));
            float4 *b = reinterpret_cast<float4 *>(mine + 4096 + ((j ^ sw) << 4));
            float4 xa = *a, xv = *b;
            xa.x += v0[4 * j]; xa.y += v0[4 * j + 1]; xa.z += v0[4 * j + 2]; xa.w += v0[4 * j + 3];
            xv.x += v1[4 * j]; xv.y += v1[4 * j + 1]; xv.z += v1[4 * j + 2]; xv.w += v1[4 * j + 3];
            *a = xa;
            *b = xv;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmOut, ebuf, col + c, row0);
            tma_store_2d(tmOut, ebuf + 4096, col + c + 32, row0);
            bulk_commit();
        }
    }
    return true;
}

template <int BN, int MODE>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm2(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ TmapB tmB,
            const __grid_constant__ CUtensorMap tmOut, const GemmArgs p) {
    using C = Cfg2<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + C::STAGES;
    uint64_t *tfull = empty + C::STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *xbar = drain + 1;  // per epilogue warp: its residual tile has landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xbar + EPI_WARPS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, 2 * EPI_WARPS);
        }
        mbar_init(drain, 1);
        for (int w = 0; w < EPI_WARPS; ++w) mbar_init(xbar + w, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB.m[0]);
        tma_prefetch_desc(&tmOut);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // barriers of both CTAs initialised before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        int stage = 0;
        uint32_t phase = 0, issued = 0, last_parity = 0;
        bool ok = true;
        Walk wk(p, pair, npairs);
        int tile, kb0, kb1;
        while (ok && wk.next(p, tile, kb0, kb1)) {
            const int mb = tile / p.tiles_n, nb = tile - mb * p.tiles_n;
            const int n0 = nb * BN, seg = n0 / p.seg_n, nin = n0 - seg * p.seg_n;
            const CUtensorMap *mapB = &tmB.m[seg];
            for (int kb = kb0; kb < kb1; ++kb) {
                if (*abort_flag || !mbar_wait(empty + stage, phase ^ 1u, p.ctl)) {
                    ok = false;
                    break;
                }
                uint8_t *sa = smem + stage * C::STAGE_BYTES;
                const uint32_t bar = mapa_shared(full + stage, 0);
                if (leader) mbar_arrive_expect_tx(full + stage, 2 * C::STAGE_BYTES);
                tma_load_2d_pair(sa, &tmA, bar, kb * BK, mb * 256 + (int)rank * 128);
                tma_load_2d_pair(sa + C::A_BYTES, mapB, bar, kb * BK, nin + (int)rank * (BN / 2));
                issued |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) *abort_flag = 1;
        // The even CTA's full barriers count both CTAs' bytes: once they complete, no copy of
        // either CTA is in flight.  (After a wait has run out, the teardown is >= 1 s later,
        // long after any copy has landed.)
        if (leader)
            for (int s = 0; s < C::STAGES; ++s)
                if ((issued >> s) & 1u) mbar_wait(full + s, (last_parity >> s) & 1u, p.ctl);
    } else if (warp == 1 && lane == 0 && leader) {
        // ---------------- MMA issuer (even CTA) ----------------
        constexpr uint32_t IDESC = idesc_bf16_f32(256, BN);
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool ok = true;
        Walk wk(p, pair, npairs);
        int tile, kb0, kb1;
        while (ok && wk.next(p, tile, kb0, kb1)) {
            if (*abort_flag || !mbar_wait(tempty + acc, acc_phase ^ 1u, p.ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (*abort_flag || !mbar_wait(full + stage, phase, p.ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
                const uint64_t ad = sdesc_sw128(sa), bd = sdesc_sw128(sa + C::A_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16_pair(d_tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), IDESC,
                                   (kb != kb0 || k != 0) ? 1u : 0u);
                umma_commit_pair(empty + stage, 0x3);  // frees the stage in both CTAs
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit_pair(tfull + acc, 0x3);  // accumulator ready in both CTAs
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (!ok) *abort_flag = 1;
        umma_commit_pair(drain, 0x1);
        mbar_wait(drain, 0, p.ctl);  // every MMA of this pair has completed
    } else if (warp >= 2) {
        // ---------------- epilogue (both CTAs: own 128 rows) ----------------
        // Two warps per TMEM lane quarter: warp w reads lanes 32 (w % 4) .. + 31 and one half
        // of the accumulator's columns, 64 columns per TMEM round trip.  Dense outputs go
        // through a per-warp 32 x 64 staging tile in shared memory (128-byte swizzle) and a
        // TMA store; the fp32 residual tile is brought in by TMA first and updated in place.
        constexpr bool TMA_EPI = MODE == GEMM_BF16 || MODE == GEMM_GELU_BF16 || MODE == GEMM_RESID_F32;
        const int q = warp & 3, half = (warp - 2) >> 2, ew = warp - 2;
        uint8_t *ebuf = smem + C::EPI_OFF + ew * C::EPI_BUF;
        uint64_t *xb = xbar + ew;
        uint32_t xphase = 0;
        const uint32_t tempty_leader0 = mapa_shared(tempty, 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        Walk wk(p, pair, npairs);
        int tile, kb0, kb1;
        while (wk.next(p, tile, kb0, kb1)) {
            ok = !*abort_flag && mbar_wait(tfull + acc, acc_phase, p.ctl);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int mb = tile / p.tiles_n, nb = tile - mb * p.tiles_n;
            const int row0 = mb * 256 + (int)rank * 128 + q * 32, row = row0 + lane;
            const int c0 = half * (BN / 2);
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + c0);
            if constexpr (MODE == GEMM_RESID_F32) {
                if (kb0 > 0 || kb1 < p.num_kb) {  // a stream-K piece of a tile cut by a pair boundary
                    const int slot = kb0 > 0 ? pair : pair + 1, part = kb0 > 0 ? 1 : 0;
                    ok = sk_epilogue<BN>(p, &tmB.w, &tmOut, ebuf, xb, xphase, tbase,
                                         tempty_leader0 + (uint32_t)(acc * 8), slot, part,
                                         slot * 512 + (int)rank * 128 + q * 32, row0, c0, nb * BN + c0,
                                         p.sk_tickets + (slot * 2 + (int)rank) * EPI_WARPS + ew, lane);
                    if (!ok) {
                        *abort_flag = 1;
                        break;
                    }
                    if (++acc == 2) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                    continue;
                }
            }
#pragma unroll 1
            for (int c = 0; c < BN / 2; c += 64) {
                const int col = nb * BN + c0 + c;
                if constexpr (TMA_EPI) {
                    if (lane == 0) {
                        bulk_wait_read0();  // the previous store has finished reading ebuf
                        if constexpr (MODE == GEMM_RESID_F32) {
                            fence_proxy_async_smem();
                            mbar_arrive_expect_tx(xb, 2 * 4096);
                            tma_load_2d(ebuf, &tmOut, xb, col, row0);
                            tma_load_2d(ebuf + 4096, &tmOut, xb, col + 32, row0);
                        }
                    }
                    __syncwarp();
                }
                uint32_t r0[32], r1[32];
                tmem_ld32(tbase + (uint32_t)c, r0);
                tmem_ld32(tbase + (uint32_t)c + 32u, r1);
                tmem_wait_ld();
                if (c + 64 >= BN / 2) {  // last TMEM read of this tile: hand the accumulator back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(tempty_leader0 + (uint32_t)(acc * 8));
                }
                if constexpr (TMA_EPI) {
                    float v0[32], v1[32];
                    bias_act<MODE>(p, col, r0, v0);
                    bias_act<MODE>(p, col + 32, r1, v1);
                    uint8_t *mine = ebuf + lane * 128;
                    const int sw = lane & 7;
                    if constexpr (MODE == GEMM_RESID_F32) {
                        ok = __all_sync(0xffffffffu, mbar_wait(xb, xphase, p.ctl));
                        xphase ^= 1u;
                        if (!ok) {
                            *abort_flag = 1;
                            break;
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j) {  // 16-byte chunk j = columns 4j .. 4j+3
                            float4 *a = reinterpret_cast<float4 *>(mine + ((j ^ sw) << 4));
                            float4 *b = reinterpret_cast<float4 *>(mine + 4096 + ((j ^ sw) << 4));
                            float4 xa = *a, xv = *b;
                            xa.x += v0[4 * j]; xa.y += v0[4 * j + 1]; xa.z += v0[4 * j + 2]; xa.w += v0[4 * j + 3];
                            xv.x += v1[4 * j]; xv.y += v1[4 * j + 1]; xv.z += v1[4 * j + 2]; xv.w += v1[4 * j + 3];
                            *a = xa;
                            *b = xv;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {  // 16-byte chunk j = columns 8j .. 8j+7
                            const float *v = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
                            *reinterpret_cast<uint4 *>(mine + ((j ^ sw) << 4)) =
                                make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                                           pack_bf16(v[6], v[7]));
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (MODE == GEMM_RESID_F32) {
                            tma_store_2d(&tmOut, ebuf, col, row0);
                            tma_store_2d(&tmOut, ebuf + 4096, col + 32, row0);
                        } else {
                            tma_store_2d(&tmOut, ebuf, col, row0);
                        }
                        bulk_commit();
                    }
                } else if (row < p.M) {
                    epilogue_chunk<MODE>(p, row, col, r0);
                    epilogue_chunk<MODE>(p, row, col + 32, r1);
                }
            }
            if (!ok) break;
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait0();  // every store of this warp has completed
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still signal its barriers
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}


template <int BN, int MODE>
int launch_pair_t(const CUtensorMap &ta, const TmapB &tb, const CUtensorMap &to, const GemmArgs &a, int grid,
                  cudaStream_t s) {
    auto kern = k_gemm2<BN, MODE>;  // shared-memory attribute set once per device (gemm_prepare)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg2<BN>::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, to, a) != cudaSuccess) return WH_ECUDA;
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

// Number of CTA pairs of k_gemm2<BN, *> that can be resident at once (cached per device).
template <int BN>
int max_active_pairs(int num_sms) {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
    if (cached[dev] > 0) return cached[dev];
    auto kern = k_gemm2<BN, GEMM_BF16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg2<BN>::SMEM_BYTES) !=
        cudaSuccess)
        return num_sms / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms, 1, 1);
    cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg2<BN>::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = num_sms / 2;
    }
    cached[dev] = n;
    return n;
}

template <int BN, int MODE>
int set_attr() {
    return cudaFuncSetAttribute(k_gemm2<BN, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg2<BN>::SMEM_BYTES) == cudaSuccess
               ? WH_OK
               : WH_ECUDA;
}

template <int BN>
int launch_pair_mode(int mode, const CUtensorMap &ta, const TmapB &tb, const CUtensorMap &to, const GemmArgs &a,
                     int grid, cudaStream_t s) {
    switch (mode) {
        case GEMM_BF16: return launch_pair_t<BN, GEMM_BF16>(ta, tb, to, a, grid, s);
        case GEMM_GELU_BF16: return launch_pair_t<BN, GEMM_GELU_BF16>(ta, tb, to, a, grid, s);
        case GEMM_RESID_F32: return launch_pair_t<BN, GEMM_RESID_F32>(ta, tb, to, a, grid, s);
        case GEMM_CONV1: return launch_pair_t<BN, GEMM_CONV1>(ta, tb, to, a, grid, s);
        case GEMM_CONV2: return launch_pair_t<BN, GEMM_CONV2>(ta, tb, to, a, grid, s);
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

namespace {
int make_tmap(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *ptr, long long rows, int cols, int ld,
              int box_cols, int box_rows) {
    if (int rc = tmap_encoder_ready()) return rc;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * esize};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = g_encode(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? WH_OK : WH_EINVAL;
}
}  // namespace

// 2-D bf16 tensor map over rows x cols (row stride ld elements), box 64 x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
int make_tmap_bf16(CUtensorMap *m, const void *ptr, long long rows, int cols, int ld, int box_rows) {
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, rows, cols, ld, 64, box_rows);
}
int make_tmap_f32(CUtensorMap *m, const void *ptr, long long rows, int cols, int ld, int box_rows) {
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, rows, cols, ld, 32, box_rows);
}

int gemm_prepare(int num_sms) {
    int rc = 0;
    rc |= set_attr<256, GEMM_BF16>() | set_attr<256, GEMM_GELU_BF16>() | set_attr<256, GEMM_RESID_F32>();
    rc |= set_attr<256, GEMM_CONV1>() | set_attr<256, GEMM_CONV2>();
    rc |= set_attr<128, GEMM_BF16>() | set_attr<128, GEMM_GELU_BF16>() | set_attr<128, GEMM_RESID_F32>();
    rc |= set_attr<128, GEMM_CONV1>() | set_attr<128, GEMM_CONV2>();
    if (rc) return WH_ECUDA;
    max_active_pairs<256>(num_sms);
    max_active_pairs<128>(num_sms);
    return tmap_encoder_ready();
}

int gemm_launch(const GemmDesc &g, int mode, const DevCtl &ctl, int num_sms, cudaStream_t s) {
    if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.seg_n <= 0 || g.N % g.seg_n != 0 || g.N / g.seg_n > 3 ||
        g.seg_n % 128 != 0 || g.K % 8 != 0 || g.lda % 8 != 0 || g.ldb % 8 != 0)
        return WH_EINVAL;
    const int BN = (g.seg_n % 256 == 0) ? 256 : 128;
    const int nseg = g.N / g.seg_n;
    CUtensorMap ta;
    TmapB tb;
    // CTA pairs: each CTA loads 128 rows of A and BN/2 rows of B per k-block.
    if (int rc = make_tmap_bf16(&ta, g.a, g.M, g.K, g.lda, 128)) return rc;
    for (int i = 0; i < 3; ++i) {
        const void *b = g.b[i < nseg ? i : 0];
        if (int rc = make_tmap_bf16(&tb.m[i], b, g.seg_n, g.K, g.ldb, BN / 2)) return rc;
    }
    GemmArgs a;
    a.M = g.M;
    a.N = g.N;
    a.num_kb = (g.K + BK - 1) / BK;
    a.tiles_n = g.N / BN;
    const int tiles_m = (g.M + 255) / 256;  // 256-row tiles per CTA pair
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
    // Output tensor map for the TMA-store epilogues (32-row boxes); the conv modes write
    // directly and get a placeholder copy of the A map.
    CUtensorMap to = ta;
    if (mode == GEMM_BF16 || mode == GEMM_GELU_BF16) {
        if (int rc = make_tmap_bf16(&to, g.out, g.M, (int)g.ldo, (int)g.ldo, 32)) return rc;
    } else if (mode == GEMM_RESID_F32) {
        if (int rc = make_tmap_f32(&to, g.out, g.M, (int)g.ldo, (int)g.ldo, 32)) return rc;
    }
    const int resident = BN == 256 ? max_active_pairs<256>(num_sms) : max_active_pairs<128>(num_sms);
    const int pairs = a.num_tiles < resident ? a.num_tiles : resident;
    // Stream-K for the residual mode when the tiles do not fill whole rounds: every pair's share
    // (at least one tile's k-blocks, so a cut tile has exactly two pieces) ends within one tile
    // of every other pair's, instead of some pairs running one tile more than the rest.
    a.sk = 0;
    a.sk_first = 0;
    a.sk_total = 0;
    a.sk_tickets = g.sk_tickets;
    tb.w = tb.m[0];
    // Only for long k-loops (fc2): with a short one (out_proj, K = d) the two partial writes and
    // the second piece's reloads cost more than the balance saves.
    if (mode == GEMM_RESID_F32 && g.sk_ws != nullptr && g.sk_tickets != nullptr && a.num_tiles > pairs &&
        a.num_tiles % pairs != 0 && a.num_kb >= GEMM_SK_MIN_KB && pairs + 1 <= g.sk_slots &&
        g.sk_slots <= GEMM_SK_SLOTS) {
        // whole rounds but the last go round-robin (neighbouring pairs on neighbouring tiles, so
        // operands are shared in L2); the last whole round and the remainder are shared out,
        // at least one tile's k-blocks per pair
        const int first = (a.num_tiles / pairs - 1) * pairs;
        const long long total = (long long)(a.num_tiles - first) * a.num_kb;
        if (total / pairs >= a.num_kb) {
            if (int rc = make_tmap_f32(&tb.w, g.sk_ws, (long long)g.sk_slots * 512, BN, BN, 32)) return rc;
            a.sk = 1;
            a.sk_first = first;
            a.sk_total = total;
        }
    }
    count_launch();
    return BN == 256 ? launch_pair_mode<256>(mode, ta, tb, to, a, 2 * pairs, s)
                     : launch_pair_mode<128>(mode, ta, tb, to, a, 2 * pairs, s);
}

}  // namespace wh
