// Conv-stem operand preparation ("whisper 0.9.0 API", model.nu: conv1 k=3 s=1 pad=1,
// conv2 k=3 s=2 pad=1, zero padding) and the bounded-wait self-test kernel.
//
// Both convolutions run as GEMMs on the tensor cores with the K index ordered tap-major:
// column j * C + i of an im2col row holds input channel i at tap j.  For conv1 that row is
// [mel[t-1] | mel[t] | mel[t+1]] (zeros outside the window) -- built here, converted to bf16.
// conv2's im2col matrix is written directly by conv1's GEMM epilogue.  The Conv1d weights
// [c_out][c_in][3] are repacked once per call to the matching [c_out][3][c_in] order.
#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

constexpr int N_FRAMES = 3000;

// a1[b * F + t][j * M + i] = mel[b][t + j - 1][i] for the first F = n_frames frames of each
// window (0 outside 0..F-1: the encoder's zero padding at both ends of the span it reads;
// windows stay 3000 frames apart in mel), 8 columns per thread.
__global__ void __launch_bounds__(256) k_mel_im2col(const float *__restrict__ mel, int batch, int n_mels,
                                                    int n_frames, uint4 *__restrict__ a1) {
    const int groups_per_row = 3 * n_mels / 8;
    const long long total = (long long)batch * n_frames * groups_per_row;
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
         it += (long long)gridDim.x * blockDim.x) {
        const long long row = it / groups_per_row;
        const int gcol = (int)(it - row * groups_per_row) * 8;
        const int j = gcol / n_mels, i = gcol - j * n_mels;
        const int b = (int)(row / n_frames), t = (int)(row - (long long)b * n_frames) + j - 1;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (t >= 0 && t < n_frames) {
            const float4 *src = reinterpret_cast<const float4 *>(mel + ((long long)b * N_FRAMES + t) * n_mels + i);
            const float4 p = __ldg(src), q = __ldg(src + 1);
            o = make_uint4(pack_bf16(p.x, p.y), pack_bf16(p.z, p.w), pack_bf16(q.x, q.y), pack_bf16(q.z, q.w));
        }
        a1[it] = o;
    }
}

// y = bf16(x), 4 values per thread: the encoder memory as the cross-attention GEMMs' operand.
__global__ void __launch_bounds__(256) k_cast_bf16(const float4 *__restrict__ x, long long n4,
                                                   uint2 *__restrict__ y) {
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < n4;
         it += (long long)gridDim.x * blockDim.x) {
        const float4 v = __ldg(x + it);
        y[it] = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
    }
}

// wp[o][j * c_in + i] = w[o][i][j]
__global__ void __launch_bounds__(256) k_pack_conv(const uint16_t *__restrict__ w, int c_out, int c_in,
                                                   uint16_t *__restrict__ wp) {
    const long long total = (long long)c_out * c_in * 3;
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
         it += (long long)gridDim.x * blockDim.x) {
        const long long o = it / (3LL * c_in);
        const int r = (int)(it - o * 3LL * c_in);
        const int j = r / c_in, i = r - j * c_in;
        wp[it] = w[(o * c_in + i) * 3 + j];
    }
}

// One block waits on an mbarrier that nothing completes; the bounded wait runs out,
// records WH_ETIMEOUT and the block returns.
__global__ void k_selftest_timeout(DevCtl ctl) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, ctl);
    __syncthreads();
}

int grid_for(long long items) {
    long long g = (items + 255) / 256;
    return (int)(g > 8192 ? 8192 : (g < 1 ? 1 : g));
}

}  // namespace

int stem_im2col_launch(const float *mel, int batch, int n_mels, int n_frames, void *a1, cudaStream_t s) {
    if (n_frames <= 0 || n_frames > N_FRAMES) return WH_EINVAL;
    const long long items = (long long)batch * n_frames * (3 * n_mels / 8);
    k_mel_im2col<<<grid_for(items), 256, 0, s>>>(mel, batch, n_mels, n_frames, reinterpret_cast<uint4 *>(a1));
    count_launch();
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

int cast_bf16_launch(const float *x, long long n, void *y, cudaStream_t s) {
    if (n <= 0) return WH_OK;
    if (n % 4 != 0) return WH_EINVAL;
    k_cast_bf16<<<grid_for(n / 4), 256, 0, s>>>(reinterpret_cast<const float4 *>(x), n / 4,
                                                 reinterpret_cast<uint2 *>(y));
    count_launch();
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

int pack_conv_weight_launch(const void *w, int c_out, int c_in, void *wp, cudaStream_t s) {
    k_pack_conv<<<grid_for((long long)c_out * c_in * 3), 256, 0, s>>>(reinterpret_cast<const uint16_t *>(w), c_out,
                                                                     c_in, reinterpret_cast<uint16_t *>(wp));
    count_launch();
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

int selftest_timeout_launch(const DevCtl &ctl, cudaStream_t s) {
    k_selftest_timeout<<<1, 32, 0, s>>>(ctl);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

}  // namespace wh
