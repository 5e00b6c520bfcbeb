// Log-mel front end ("How Audio Becomes Words: Whisper's Kernels Step By Step On A CPU",
// section "The Frontend: Sound Becomes A Tensor", kernels 3-6 and the bullets that walk them):
// pad/truncate to 480000 samples, reflect padding, periodic Hann(400), n_fft 400, hop 160,
// power re^2 + im^2 on the 201 x 3000 grid, Slaney area-normalised mel filters, log10,
// clamp at (window maximum - 8) and (x + 4) / 4.
//
// Kernel 1 (k_logmel): one block = 30 consecutive frames of one window.  The 5040 samples
// the frames touch are staged once in shared memory (coalesced; reflect and zero-extension
// applied while loading).  Each real 400-point frame x is transformed as one complex
// 200-point FFT of z[m] = x[2m] + i x[2m+1] (decomposed 200 = 8 x 25, the 25-point part as
// 5 x 5), then split into the real spectrum X[k] = E[k] + W400^k O[k], k = 0..200.  The
// power spectrum stays in shared memory; the sparse mel projection, log10 and the block's
// maximum follow; one atomicMax per block builds the per-window maximum.
// Kernel 2 (k_clamp): mel = (max(mel, g - 8) + 4) / 4 in place with the window maximum g.
// Both read/write only the PCM and the log-mel (the intermediates never reach HBM).
#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

constexpr int N_FFT = 400, HOP = 160, N_FRAMES = 3000, N_SAMPLES = 480000, N_BINS = 201;
constexpr int FB = 30;                          // frames per block: 3000 = 100 x 30
constexpr int THREADS = 256;
constexpr int SEG = FB * HOP + (N_FFT - HOP);   // 5040 staged samples
constexpr int ZSTRIDE = 200;                    // complex slots per frame
constexpr int MAXW = 512;                       // mel filter nonzeros (<= 2 per bin)
// The staged samples are dead after stage A, so the power spectrum reuses their space.
constexpr int SEGP = SEG > FB * N_BINS ? SEG : FB * N_BINS;
constexpr size_t SMEM = (size_t)SEGP * 4 + (size_t)FB * ZSTRIDE * 8;

__device__ float g_hann[N_FFT];
__device__ float2 g_tw[N_FFT];          // W400^j = (cos, -sin)(2 pi j / 400)
__device__ int g_mel_start[2][128];     // first nonzero bin of filter m
__device__ int g_mel_len[2][128];       // number of nonzero bins
__device__ int g_mel_off[2][128];       // offset of its weights in g_mel_w
__device__ float g_mel_w[2][MAXW];

__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}
__device__ __forceinline__ float2 mul_negi(float2 a) { return make_float2(a.y, -a.x); }  // -i * a

// 4-point DFT (W4 = -i).
__device__ __forceinline__ void dft4(float2 &a0, float2 &a1, float2 &a2, float2 &a3) {
    const float2 t0 = cadd(a0, a2), t1 = csub(a0, a2), t2 = cadd(a1, a3), t3 = csub(a1, a3);
    a0 = cadd(t0, t2);
    a2 = csub(t0, t2);
    a1 = cadd(t1, mul_negi(t3));
    a3 = csub(t1, mul_negi(t3));
}

// 8-point DFT in place: two 4-point DFTs of the even and odd samples, then W8 twiddles.
__device__ __forceinline__ void dft8(float2 (&a)[8]) {
    float2 e0 = a[0], e1 = a[2], e2 = a[4], e3 = a[6];
    float2 o0 = a[1], o1 = a[3], o2 = a[5], o3 = a[7];
    dft4(e0, e1, e2, e3);
    dft4(o0, o1, o2, o3);
    const float r = 0.70710678118654752f;
    o1 = make_float2(r * (o1.x + o1.y), r * (o1.y - o1.x));      // * (r, -r)
    o2 = mul_negi(o2);                                           // * (0, -1)
    o3 = make_float2(r * (o3.y - o3.x), -r * (o3.x + o3.y));     // * (-r, -r)
    a[0] = cadd(e0, o0); a[4] = csub(e0, o0);
    a[1] = cadd(e1, o1); a[5] = csub(e1, o1);
    a[2] = cadd(e2, o2); a[6] = csub(e2, o2);
    a[3] = cadd(e3, o3); a[7] = csub(e3, o3);
}

// 5-point DFT of (y0..y4) with W5 = exp(-2 pi i / 5):
//   X1,4 = y0 + c1 t1 + c2 t2 -/+ i (s1 t3 + s2 t4),  X2,3 = y0 + c2 t1 + c1 t2 -/+ i (s2 t3 - s1 t4)
// with t1 = y1 + y4, t2 = y2 + y3, t3 = y1 - y4, t4 = y2 - y3.
__device__ __forceinline__ void dft5(float2 &y0, float2 &y1, float2 &y2, float2 &y3, float2 &y4) {
    const float c1 = 0.30901699437494742f, c2 = -0.80901699437494742f;
    const float s1 = 0.95105651629515357f, s2 = 0.58778525229247313f;
    const float2 t1 = cadd(y1, y4), t2 = cadd(y2, y3), t3 = csub(y1, y4), t4 = csub(y2, y3);
    const float2 a = make_float2(y0.x + c1 * t1.x + c2 * t2.x, y0.y + c1 * t1.y + c2 * t2.y);
    const float2 b = make_float2(y0.x + c2 * t1.x + c1 * t2.x, y0.y + c2 * t1.y + c1 * t2.y);
    const float2 u = make_float2(s1 * t3.x + s2 * t4.x, s1 * t3.y + s2 * t4.y);
    const float2 w = make_float2(s2 * t3.x - s1 * t4.x, s2 * t3.y - s1 * t4.y);
    y0 = make_float2(y0.x + t1.x + t2.x, y0.y + t1.y + t2.y);
    y1 = cadd(a, mul_negi(u));
    y4 = csub(a, mul_negi(u));
    y2 = cadd(b, mul_negi(w));
    y3 = csub(b, mul_negi(w));
}

// Order-preserving map float -> uint32 (for atomicMax over signed floats).
__device__ __forceinline__ uint32_t f2key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Window b starts at pcm + b * stride and holds min(n, total - b * stride) samples (a batch of
// clips: stride = n, total = batch * n; one long clip cut into 30-s windows: stride = n =
// 480000, total = the clip's length).
__global__ void __launch_bounds__(THREADS) k_logmel(const float *__restrict__ pcm, long long n, long long stride,
                                                    long long total, int n_mels, int table,
                                                    float *__restrict__ mel, uint32_t *__restrict__ wmax) {
    extern __shared__ float4 smem4[];
    float *seg = reinterpret_cast<float *>(smem4);       // staged samples, then the power [FB][201]
    float2 *Z = reinterpret_cast<float2 *>(seg + SEGP);  // [FB][ZSTRIDE]
    float *P = seg;
    __shared__ float red[THREADS / 32];

    const int tid = threadIdx.x;
    const int b = blockIdx.y;
    const int t0 = blockIdx.x * FB;
    const int nf = min(FB, N_FRAMES - t0);
    const float *x = pcm + (long long)b * stride;
    n = min(n, total - (long long)b * stride);

    // Stage samples 160 t0 - 200 ... (pad/truncate to 480000, then reflect by 200).  Blocks
    // whose span lies inside the clip and is 16-byte aligned copy with float4 loads.
    const long long s0 = (long long)HOP * t0 - N_FFT / 2;
    const long long lim = n < N_SAMPLES ? n : N_SAMPLES;
    if (s0 >= 0 && s0 + SEG <= lim && ((reinterpret_cast<uintptr_t>(x + s0) & 15) == 0)) {
        const float4 *src = reinterpret_cast<const float4 *>(x + s0);
        float4 *dst = reinterpret_cast<float4 *>(seg);
        for (int j = tid; j < SEG / 4; j += THREADS) dst[j] = __ldg(src + j);
    } else {
        for (int j = tid; j < SEG; j += THREADS) {
            int si = (int)s0 + j;
            si = si < 0 ? -si : si;
            si = si > N_SAMPLES - 1 ? 2 * (N_SAMPLES - 1) - si : si;
            seg[j] = (si < n) ? __ldg(x + si) : 0.0f;
        }
    }
    __syncthreads();

    // Stage A: for each frame f and n2 in 0..24, the 8-point DFT over n1 of z[25 n1 + n2]
    // (z[m] = w[2m] x[2m] + i w[2m+1] x[2m+1]), times W200^(n2 k1); stored as Z[f][25 k1 + n2].
    for (int it = tid; it < nf * 25; it += THREADS) {
        const int f = it / 25, n2 = it - f * 25;
        const float *xf = seg + f * HOP;
        float2 a[8];
#pragma unroll
        for (int n1 = 0; n1 < 8; ++n1) {
            const int m = 25 * n1 + n2;
            a[n1] = make_float2(g_hann[2 * m] * xf[2 * m], g_hann[2 * m + 1] * xf[2 * m + 1]);
        }
        dft8(a);
        float2 *zf = Z + f * ZSTRIDE;
        zf[n2] = a[0];
#pragma unroll
        for (int k1 = 1; k1 < 8; ++k1) zf[25 * k1 + n2] = cmul(a[k1], g_tw[2 * n2 * k1]);
    }
    __syncthreads();

    // Stage B: for each frame f and k1 in 0..7, the 25-point DFT over n2 (n2 = 5a + b,
    // k2 = c + 5e): 5-point DFTs over a, twiddles W25^(b c), 5-point DFTs over b.
    // Output Z200[k1 + 8 k2] is written back in natural order after a block barrier.
    float2 y[25];
    int fB = -1, k1B = 0;
    {
        const int it = tid;  // nf * 8 <= 256 items: one per thread
        if (it < nf * 8) {
            fB = it >> 3;
            k1B = it & 7;
            const float2 *col = Z + fB * ZSTRIDE + 25 * k1B;
#pragma unroll
            for (int i = 0; i < 25; ++i) y[i] = col[i];
#pragma unroll
            for (int bb = 0; bb < 5; ++bb) dft5(y[bb], y[5 + bb], y[10 + bb], y[15 + bb], y[20 + bb]);
            // now y[5 c + bb] = U[bb][c]
#pragma unroll
            for (int bb = 1; bb < 5; ++bb)
#pragma unroll
                for (int c = 1; c < 5; ++c) y[5 * c + bb] = cmul(y[5 * c + bb], g_tw[16 * bb * c]);
#pragma unroll
            for (int c = 0; c < 5; ++c) dft5(y[5 * c], y[5 * c + 1], y[5 * c + 2], y[5 * c + 3], y[5 * c + 4]);
            // now y[5 c + e] = Z25[c + 5 e]
        }
    }
    __syncthreads();
    if (fB >= 0) {
        float2 *zf = Z + fB * ZSTRIDE;
#pragma unroll
        for (int c = 0; c < 5; ++c)
#pragma unroll
            for (int e = 0; e < 5; ++e) zf[k1B + 8 * (c + 5 * e)] = y[5 * c + e];
    }
    __syncthreads();

    // Stage C: real spectrum and power, one warp per frame, lanes over bins.
    // E = (Z[k] + conj Z[-k]) / 2, O = -i (Z[k] - conj Z[-k]) / 2, X[k] = E + W400^k O, P = |X|^2.
    const int warp = tid >> 5, lane = tid & 31;
    for (int f = warp; f < nf; f += THREADS / 32) {
        const float2 *zf = Z + f * ZSTRIDE;
        float *pf = P + f * N_BINS;
        for (int k = lane; k < N_BINS; k += 32) {
            const float2 zk = zf[k == 200 ? 0 : k];
            const float2 zm = zf[k == 0 ? 0 : 200 - k];
            const float2 e = make_float2(0.5f * (zk.x + zm.x), 0.5f * (zk.y - zm.y));
            const float2 o = make_float2(0.5f * (zk.y + zm.y), -0.5f * (zk.x - zm.x));
            const float2 X = cadd(e, cmul(g_tw[k], o));
            pf[k] = X.x * X.x + X.y * X.y;
        }
    }
    __syncthreads();

    // Stage D: mel projection, log10 with floor 1e-10, frame-major store, block maximum.
    // One warp per frame, lanes over mel bins (coalesced stores).
    float lmax = -INFINITY;
    const int *mstart = g_mel_start[table], *mlen = g_mel_len[table], *moff = g_mel_off[table];
    const float *mw = g_mel_w[table];
    for (int f = warp; f < nf; f += THREADS / 32) {
        const float *pf = P + f * N_BINS;
        float *out = mel + ((long long)b * N_FRAMES + t0 + f) * n_mels;
        for (int m = lane; m < n_mels; m += 32) {
            const int k0 = mstart[m], len = mlen[m];
            const float *wm = mw + moff[m];
            float acc = 0.0f;
            for (int i = 0; i < len; ++i) acc = fmaf(wm[i], pf[k0 + i], acc);
            // log10 via the hardware log2 (log10 x = log2 x * log10 2); at the floor exactly -10.
            float lg2;
            asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg2) : "f"(acc));
            const float lg = acc > 1e-10f ? lg2 * 0.30102999566398120f : -10.0f;
            out[m] = lg;
            lmax = fmaxf(lmax, lg);
        }
    }
    lmax = warp_max(lmax);
    if (lane == 0) red[warp] = lmax;
    __syncthreads();
    if (tid < 32) {
        float v = tid < THREADS / 32 ? red[tid] : -INFINITY;
        v = warp_max(v);
        if (tid == 0) atomicMax(wmax + b, f2key(v));
    }
}

// grid.y = window: mel[b] = (max(mel[b], g_b - 8) + 4) / 4, float4 at a time.
__global__ void __launch_bounds__(256) k_clamp(float4 *__restrict__ mel, int per_window4,
                                               const uint32_t *__restrict__ wmax) {
    const int b = blockIdx.y;
    const float floor = key2f(wmax[b]) - 8.0f;
    float4 *w = mel + (long long)b * per_window4;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < per_window4; i += gridDim.x * blockDim.x) {
        float4 v = w[i];
        v.x = (fmaxf(v.x, floor) + 4.0f) * 0.25f;
        v.y = (fmaxf(v.y, floor) + 4.0f) * 0.25f;
        v.z = (fmaxf(v.z, floor) + 4.0f) * 0.25f;
        v.w = (fmaxf(v.w, floor) + 4.0f) * 0.25f;
        w[i] = v;
    }
}

// ---- host-side constant tables (built in double precision) ----------------------------
double hz_to_mel(double f) {  // Slaney: 3 f / 200 below 1 kHz, 27 mel per factor 6.4 above
    return f < 1000.0 ? 3.0 * f / 200.0 : 15.0 + 27.0 * std::log(f / 1000.0) / std::log(6.4);
}
double mel_to_hz(double m) {
    return m < 15.0 ? 200.0 * m / 3.0 : 1000.0 * std::exp((m - 15.0) * std::log(6.4) / 27.0);
}

struct MelTable {
    int start[128], len[128], off[128];
    float w[MAXW];
};

int build_mel(int n_mels, MelTable &t) {
    const double top = hz_to_mel(8000.0);
    std::vector<double> f(n_mels + 2);
    for (int i = 0; i < n_mels + 2; ++i) f[i] = mel_to_hz(top * i / (n_mels + 1));
    int used = 0;
    for (int m = 0; m < n_mels; ++m) {
        const double lo = f[m], c = f[m + 1], hi = f[m + 2], norm = 2.0 / (hi - lo);
        int k0 = -1, k1 = -1;
        for (int k = 0; k < N_BINS; ++k) {
            const double fk = 40.0 * k;
            const double v = std::fmax(0.0, std::fmin((fk - lo) / (c - lo), (hi - fk) / (hi - c)));
            if (v > 0.0) {
                if (k0 < 0) k0 = k;
                k1 = k;
            }
        }
        if (k0 < 0) {  // empty filter (cannot happen for 80 or 128 bins): one zero weight
            k0 = 0;
            k1 = 0;
        }
        t.start[m] = k0;
        t.len[m] = k1 - k0 + 1;
        t.off[m] = used;
        if (used + t.len[m] > MAXW) return WH_EINVAL;
        for (int k = k0; k <= k1; ++k) {
            const double fk = 40.0 * k;
            const double v = std::fmax(0.0, std::fmin((fk - lo) / (c - lo), (hi - fk) / (hi - c)));
            t.w[used++] = (float)(v * norm);
        }
    }
    return WH_OK;
}

}  // namespace

int frontend_init_tables() {
    float hann[N_FFT];
    float2 tw[N_FFT];
    const double pi = 3.14159265358979323846;
    for (int j = 0; j < N_FFT; ++j) {
        hann[j] = (float)(0.5 - 0.5 * std::cos(2.0 * pi * j / N_FFT));
        tw[j] = make_float2((float)std::cos(2.0 * pi * j / N_FFT), (float)-std::sin(2.0 * pi * j / N_FFT));
    }
    static MelTable mt[2];
    static std::once_flag once;
    static int build_rc = WH_OK;
    std::call_once(once, [] {
        build_rc = build_mel(80, mt[0]);
        if (build_rc == WH_OK) build_rc = build_mel(128, mt[1]);
    });
    if (build_rc != WH_OK) return build_rc;
    int start[2][128], len[2][128], off[2][128];
    float w[2][MAXW];
    for (int t = 0; t < 2; ++t) {
        for (int m = 0; m < 128; ++m) {
            start[t][m] = mt[t].start[m];
            len[t][m] = mt[t].len[m];
            off[t][m] = mt[t].off[m];
        }
        for (int i = 0; i < MAXW; ++i) w[t][i] = mt[t].w[i];
    }
    if (cudaMemcpyToSymbol(g_hann, hann, sizeof(hann)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_tw, tw, sizeof(tw)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_mel_start, start, sizeof(start)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_mel_len, len, sizeof(len)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_mel_off, off, sizeof(off)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_mel_w, w, sizeof(w)) != cudaSuccess)
        return WH_ECUDA;
    if (cudaFuncSetAttribute(k_logmel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) != cudaSuccess)
        return WH_ECUDA;
    return WH_OK;
}

int frontend_launch(const float *pcm, int64_t n, int64_t stride, int64_t total, int batch, int n_mels, float *mel,
                    uint32_t *wmax, cudaStream_t s) {
    if (cudaMemsetAsync(wmax, 0, sizeof(uint32_t) * (size_t)batch, s) != cudaSuccess) return WH_ECUDA;
    dim3 grid((N_FRAMES + FB - 1) / FB, batch);
    k_logmel<<<grid, THREADS, SMEM, s>>>(pcm, (long long)n, (long long)stride, (long long)total, n_mels,
                                         n_mels == 128 ? 1 : 0, mel, wmax);
    const int per4 = N_FRAMES * n_mels / 4;
    dim3 cgrid((per4 + 255) / 256, batch);
    k_clamp<<<cgrid, 256, 0, s>>>(reinterpret_cast<float4 *>(mel), per4, wmax);
    count_launch(2);
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

}  // namespace wh
