// Resampling of PCM to 16 kHz with a windowed-sinc polyphase filter ("whisper" package page,
// "Transcribing": input at any sample rate is resampled to 16 kHz with a windowed sinc, not
// by linear interpolation; "How it is verified": the resampler is checked against scipy's
// resample_poly).  The filter is resample_poly's default design, restated:
//   up / down = 16000 / rate_in in lowest terms, M = max(up, down), H = 10 M,
//   h[t] = up * w[t] * f sinc(f (t - H)) / S,   t = 0 .. 2H,   f = 1 / M,
//   w = Kaiser window (beta 5) over the 2H + 1 taps, S = sum_t w[t] f sinc(f (t - H))
//   (unit gain at DC before the factor up), and
//   y[j] = sum_i h[j down + H - i up] x[i],   j = 0 .. ceil(n up / down) - 1,
// i.e. the signal upsampled by `up`, low-pass filtered (zero phase) and kept every `down`-th
// sample.  The filter is split into `up` phases of K = ceil((2H + 1) / up) taps:
// P[p][k] = h[p + k up], so output j uses phase p = (j down + H) mod up against the K input
// samples i_hi, i_hi - 1, ... with i_hi = floor((j down + H) / up).
//
// k_resample_table builds P on the device in float64 (S is summed once per rate on the host),
// so a call records into a CUDA graph without host-to-device copies; k_resample computes one
// output sample per thread from a block-wide input span staged in shared memory.
#include <cmath>
#include <map>
#include <mutex>
#include <numeric>

#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

constexpr double KAISER_BETA = 5.0;
constexpr int TARGET_RATE = 16000;

struct Plan {
    long long up, down, M, H, K;
};

Plan plan_of(int rate_in) {
    const long long g = std::gcd((long long)TARGET_RATE, (long long)rate_in);
    Plan p;
    p.up = TARGET_RATE / g;
    p.down = rate_in / g;
    p.M = p.up > p.down ? p.up : p.down;
    p.H = 10 * p.M;
    p.K = (2 * p.H + 1 + p.up - 1) / p.up;
    return p;
}

// Modified Bessel function of the first kind, order 0, by its power series
// sum_k ((x/2)^2)^k / (k!)^2 (all terms positive; |x| <= 5 here, so 40 terms are ample).
__host__ __device__ double bessel_i0(double x) {
    const double q = 0.25 * x * x;
    double term = 1.0, sum = 1.0;
    for (int k = 1; k < 60; ++k) {
        term *= q / ((double)k * (double)k);
        sum += term;
        if (term < 1e-18 * sum) break;
    }
    return sum;
}

__host__ __device__ double kaiser(long long t, long long H) {
    const double r = (double)(t - H) / (double)H;
    const double a = 1.0 - r * r;
    return bessel_i0(KAISER_BETA * sqrt(a > 0.0 ? a : 0.0)) / bessel_i0(KAISER_BETA);
}

// f sinc(f (t - H)) with sinc(x) = sin(pi x) / (pi x)
double lowpass_host(long long t, long long H, double f) {
    const double x = f * (double)(t - H);
    if (x == 0.0) return f;
    const double pi = 3.14159265358979323846;
    return f * std::sin(pi * x) / (pi * x);
}

__global__ void k_resample_table(Plan pl, double inv_s, float *__restrict__ table) {
    const long long n = pl.up * pl.K;
    const double f = 1.0 / (double)pl.M;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long p = idx / pl.K, k = idx - p * pl.K;
        const long long t = p + k * pl.up;
        double h = 0.0;
        if (t <= 2 * pl.H) {
            const double x = f * (double)(t - pl.H);
            const double lp = (x == 0.0) ? f : f * sinpi(x) / (3.14159265358979323846 * x);
            h = (double)pl.up * kaiser(t, pl.H) * lp * inv_s;
        }
        table[idx] = (float)h;
    }
}

// A block computes tiles of 256 consecutive outputs.  Their taps read one contiguous input
// span, staged in shared memory first (zeros outside the clip), so the inner loop is a plain
// FMA chain over the phase's K taps: xs[ihi - lo - k] * P[p][k].  Consecutive outputs use
// different phases, so when the table fits (SMEM_TABLE) the block first copies it into shared
// memory with an odd row stride (lanes of a warp then hit distinct banks) and walks many
// tiles; larger tables (input rates with few common factors with 16 kHz) are read through L1.
constexpr int RS_THREADS = 256;
constexpr size_t RS_TABLE_SMEM_MAX = 40 * 1024;

template <bool SMEM_TABLE>
__global__ void __launch_bounds__(RS_THREADS) k_resample(const float *__restrict__ x, long long n_in, Plan pl,
                                                         const float *__restrict__ table, float *__restrict__ y,
                                                         long long n_out, int span) {
    extern __shared__ float sm_rs[];
    const int K = (int)pl.K;
    const int ks = SMEM_TABLE ? (K | 1) : K;   // table row stride
    float *tab = sm_rs;                        // [up][ks] when SMEM_TABLE
    float *xs = sm_rs + (SMEM_TABLE ? (int)pl.up * ks : 0);
    if (SMEM_TABLE) {
        const int n = (int)pl.up * K;
        for (int t = threadIdx.x; t < n; t += RS_THREADS) {
            const int pp = t / K, kk = t - pp * K;
            tab[pp * ks + kk] = __ldg(table + t);
        }
    }
    const float *tp = SMEM_TABLE ? tab : table;
    const float *xb = x + (long long)blockIdx.y * n_in;
    float *yb = y + (long long)blockIdx.y * n_out;
    for (long long j0 = (long long)blockIdx.x * RS_THREADS; j0 < n_out; j0 += (long long)gridDim.x * RS_THREADS) {
        const long long jl = j0 + RS_THREADS - 1 < n_out ? j0 + RS_THREADS - 1 : n_out - 1;
        const long long ihi0 = (j0 * pl.down + pl.H) / pl.up, ihi1 = (jl * pl.down + pl.H) / pl.up;
        const long long lo = ihi0 - (K - 1);
        const int cnt = (int)(ihi1 - lo + 1);   // <= span (the launch's bound)
        __syncthreads();                        // the table is in; the previous tile's reads are done
        for (int t = threadIdx.x; t < cnt && t < span; t += RS_THREADS) {
            const long long i = lo + t;
            xs[t] = (i >= 0 && i < n_in) ? __ldg(xb + i) : 0.0f;
        }
        __syncthreads();
        const long long j = j0 + threadIdx.x;
        if (j < n_out) {
            const long long m = j * pl.down + pl.H;
            const long long ihi = m / pl.up;
            const float *ph = tp + (m - ihi * pl.up) * ks;
            const float *xp = xs + (ihi - lo);
            float acc = 0.0f;
#pragma unroll 4
            for (int k = 0; k < K; ++k) acc = fmaf(ph[k], xp[-k], acc);
            yb[j] = acc;
        }
    }
}

size_t table_smem_bytes(const Plan &pl) { return (size_t)pl.up * (size_t)(pl.K | 1) * sizeof(float); }
size_t span_of(const Plan &pl) { return (size_t)((RS_THREADS - 1) * pl.down / pl.up + 1 + pl.K + 1); }

std::mutex g_norm_mu;
std::map<int, double> g_norm;   // S per input rate

double norm_of(int rate_in, const Plan &pl) {
    std::lock_guard<std::mutex> lk(g_norm_mu);
    auto it = g_norm.find(rate_in);
    if (it != g_norm.end()) return it->second;
    const double f = 1.0 / (double)pl.M;
    double s = 0.0;
    for (long long t = 0; t <= 2 * pl.H; ++t) s += kaiser(t, pl.H) * lowpass_host(t, pl.H, f);
    g_norm[rate_in] = s;
    return s;
}

}  // namespace

void resample_forget() {
    std::lock_guard<std::mutex> lk(g_norm_mu);
    g_norm.clear();
}

bool resample_rate_ok(int rate_in) { return rate_in >= 1000 && rate_in <= 384000; }

long long resample_length(long long n_in, int rate_in) {
    const Plan pl = plan_of(rate_in);
    return (n_in * pl.up + pl.down - 1) / pl.down;
}

size_t resample_workspace(int rate_in) {
    const Plan pl = plan_of(rate_in);
    return (size_t)(pl.up * pl.K) * sizeof(float);
}

int resample_prepare() {
    // the largest dynamic shared memory a launch below asks for: a 40 KB table + a 26.4 KB span
    const int bytes = (int)(RS_TABLE_SMEM_MAX + 28 * 1024);
    return (cudaFuncSetAttribute(k_resample<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
            cudaFuncSetAttribute(k_resample<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess)
               ? WH_OK
               : WH_ECUDA;
}

int resample_launch(const float *x, long long n_in, int batch, int rate_in, float *y, void *table, int num_sms,
                    cudaStream_t s) {
    const Plan pl = plan_of(rate_in);
    const double S = norm_of(rate_in, pl);
    const long long nt = pl.up * pl.K;
    const long long tb = (nt + 255) / 256;
    k_resample_table<<<(unsigned)(tb < 4096 ? tb : 4096), 256, 0, s>>>(pl, 1.0 / S, static_cast<float *>(table));
    const long long n_out = resample_length(n_in, rate_in);
    int launches = 1;
    if (n_out > 0) {
        const long long tiles = (n_out + RS_THREADS - 1) / RS_THREADS;
        const size_t span = span_of(pl);
        if (span * sizeof(float) > 28 * 1024) return WH_EINVAL;   // not reached for 1 kHz .. 384 kHz
        const bool smem_table = table_smem_bytes(pl) <= RS_TABLE_SMEM_MAX;
        if (smem_table) {
            // about four blocks per SM over the whole batch (each copies the table once; up to
            // 40 + 28 KB of shared memory per block leaves room for four)
            long long per_clip = (4LL * num_sms + batch - 1) / batch;
            if (per_clip > tiles) per_clip = tiles;
            if (per_clip < 1) per_clip = 1;
            k_resample<true><<<dim3((unsigned)per_clip, batch), RS_THREADS, table_smem_bytes(pl) + span * sizeof(float),
                               s>>>(x, n_in, pl, static_cast<const float *>(table), y, n_out, (int)span);
        } else {
            k_resample<false><<<dim3((unsigned)(tiles < 8192 ? tiles : 8192), batch), RS_THREADS,
                                span * sizeof(float), s>>>(x, n_in, pl, static_cast<const float *>(table), y, n_out,
                                                          (int)span);
        }
        ++launches;
    }
    count_launch(launches);
    return cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

}  // namespace wh
