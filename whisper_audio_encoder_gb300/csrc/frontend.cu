// Log-mel front end ("How Audio Becomes Words: Whisper's Kernels Step By Step On A CPU",
// section "The Frontend: Sound Becomes A Tensor", kernels 3-6 and the bullets that walk them):
// pad/truncate to 480000 samples, reflect padding, periodic Hann(400), n_fft 400, hop 160,
// power re^2 + im^2 on the 201 x 3000 grid, Slaney area-normalised mel filters, log10,
// clamp at (window maximum - 8) and (x + 4) / 4.
//
// k_logmel: a persistent grid; one block transforms a tile of 32 consecutive frames of one
// window at a time, one frame per lane.  The 5360 samples the tile touches are staged once in shared memory (coalesced;
// reflect and zero-extension applied while loading), two pad floats after every 160 samples
// so that the 32 frames' rows start in distinct banks.  Each real 400-point frame x is
// transformed as the complex 200-point FFT of z[m] = w[2m] x[2m] + i w[2m+1] x[2m+1] (w the
// Hann window), split by the prime-factor (Good-Thomas) map 200 = 8 x 25: with
// m = (25 n1 + 8 n2) mod 200 and k = (25 k1 + 176 k2) mod 200,
//   Z[k] = sum_n2 W25^(n2 k2) sum_n1 W8^(n1 k1) z[m],
// i.e. 8-point DFTs over n1 then 25-point DFTs (5 x 5) over n2, with no twiddles between the
// two (8 and 25 are coprime).  The real spectrum X[k] = E[k] + W400^k O[k] (E, O the spectra
// of the even and odd samples) and its power follow, two mirrored bins (k, 200 - k) at a
// time; then the sparse mel projection, log10 and the tile's maximum; one atomicMax per tile
// builds the per-window maximum.  Every stage keeps lanes on frames and the warp on one
// index of the transform, so shared-memory accesses are conflict-free and the constant
// tables (window, gather offsets, W400^k, mel filters) are read at warp-uniform addresses.
// After a grid-wide barrier the same grid clamps: mel = (max(mel, g - 8) + 4) / 4 in place with
// the window maximum g.  Only the PCM and the log-mel touch global memory (the intermediates
// never leave shared memory).
#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace wh {

namespace {

constexpr int N_FFT = 400, HOP = 160, N_FRAMES = 3000, N_SAMPLES = 480000, N_BINS = 201;
constexpr int TF = 32;                            // frames per tile: one per lane
constexpr int THREADS = 256;
constexpr int NWARP = THREADS / 32;
constexpr int N1 = 8, N2 = 25;                    // 200 = N1 x N2
constexpr int SPAN = TF * HOP + (N_FFT - HOP);    // 5360 samples a tile touches
constexpr int ROW = HOP + 2;                      // staged floats per frame row
// Staged sample j of the span sits at j + 2 floor(j / 160).
__host__ __device__ constexpr int seg_pos(int j) { return j + 2 * (j / HOP); }
constexpr int SEG_FLOATS = seg_pos(SPAN - 1) + 2;
constexpr int P_ROWS = N_BINS - 2;                // bins 1 .. 199 (no mel filter touches 0 or 200)
constexpr int P_FLOATS = P_ROWS * TF;
constexpr int R1_FLOATS = SEG_FLOATS > P_FLOATS ? SEG_FLOATS : P_FLOATS;
constexpr int R2_FLOAT2 = N1 * N2 * TF;           // the 200-point spectra of the tile
constexpr int MT_STRIDE = 129;                    // log-mel tile row (odd: conflict-free)
constexpr int MAXW = 512;                         // mel filter nonzeros (<= 2 per bin)
constexpr size_t SMEM = (size_t)R1_FLOATS * 4 + (size_t)R2_FLOAT2 * 8;
constexpr int A_TABLE = (SEG_FLOATS + 3) / 4 * 4;  // stage-A table above the staged samples
constexpr int TILES = (N_FRAMES + TF - 1) / TF;    // tiles per window
constexpr int PF = (SPAN / 4 + THREADS - 1) / THREADS;  // prefetched float4 per thread
static_assert(A_TABLE + N2 * 24 <= R1_FLOATS, "stage-A table must fit beside the samples");
static_assert(TF * MT_STRIDE <= 2 * R2_FLOAT2, "log-mel tile must fit the spectrum region");
static_assert((R1_FLOATS * 4) % 16 == 0, "spectrum region alignment");

// Per n2, for n1 = 0 .. 7 and m = (25 n1 + 8 n2) mod 200: the Hann window pair (w[2m], w[2m+1])
// and the staged offset of sample 2m within a frame row.
struct ARow {
    float2 w[8];
    int off[8];
};
__constant__ ARow c_arow[N2];
__constant__ float2 c_tw[101];          // W400^k = (cos, -sin)(2 pi k / 400), k = 0 .. 100
__constant__ float c_mel_w[2][MAXW];    // filter weights / 4 (the power is kept x 4), filter by filter

// ---- compile-time shape of the transform and of the mel filters ------------------------
// Staged offset (within a frame row) of sample 2m for z index m = (25 n1 + 8 n2) mod 200.
__host__ __device__ constexpr int a_off(int n1, int n2) { return seg_pos(2 * ((25 * n1 + 8 * n2) % 200)); }

// Natural exp and log in double by their series, evaluated by the compiler: the Slaney mel
// filter edges (hz <-> mel) below, and from them which FFT bins each filter covers, so that
// the kernel's mel projection is straight-line code.  (The weights themselves are built on
// the host and read from c_mel_w; frontend_init_tables checks that both agree on the shape.)
constexpr double kLn2 = 0.69314718055994530942;
constexpr double ct_exp(double x) {   // exp(k ln2 + r) = 2^k exp(r), |r| <= ln2 / 2, Taylor
    int k = (int)(x / kLn2 + (x >= 0.0 ? 0.5 : -0.5));
    const double r = x - k * kLn2;
    double term = 1.0, sum = 1.0;
    for (int i = 1; i < 30; ++i) {
        term *= r / i;
        sum += term;
    }
    for (; k > 0; --k) sum *= 2.0;
    for (; k < 0; ++k) sum *= 0.5;
    return sum;
}
constexpr double ct_log(double x) {   // x = 2^e y, y in [1, 2): ln y = 2 atanh((y - 1) / (y + 1))
    int e = 0;
    while (x >= 2.0) {
        x *= 0.5;
        ++e;
    }
    while (x < 1.0) {
        x *= 2.0;
        --e;
    }
    const double z = (x - 1.0) / (x + 1.0), z2 = z * z;
    double p = z, sum = 0.0;
    for (int i = 0; i < 40; ++i) {
        sum += p / (2 * i + 1);
        p *= z2;
    }
    return 2.0 * sum + e * kLn2;
}
constexpr double ct_hz_to_mel(double f) {
    return f < 1000.0 ? 3.0 * f / 200.0 : 15.0 + 27.0 * ct_log(f / 1000.0) / ct_log(6.4);
}
constexpr double ct_mel_to_hz(double m) {
    return m < 15.0 ? 200.0 * m / 3.0 : 1000.0 * ct_exp((m - 15.0) * ct_log(6.4) / 27.0);
}

// Filter m covers the bins k with f_m < 40 k < f_(m+2) (f_i the i-th of NM + 2 edges equally
// spaced in mel from 0 to 8 kHz); its weights sit at c_mel_w[..][off[m] ...].
template <int NM>
struct MelShape {
    int start[NM], len[NM], off[NM];
    constexpr MelShape() : start(), len(), off() {
        const double top = ct_hz_to_mel(8000.0);
        int used = 0;
        for (int m = 0; m < NM; ++m) {
            const double lo = ct_mel_to_hz(top * m / (NM + 1)), hi = ct_mel_to_hz(top * (m + 2) / (NM + 1));
            int k0 = -1, k1 = -1;
            for (int k = 0; k < N_BINS; ++k) {
                const double fk = 40.0 * k;
                if (fk > lo && fk < hi) {
                    if (k0 < 0) k0 = k;
                    k1 = k;
                }
            }
            start[m] = k0;
            len[m] = k0 < 0 ? 0 : k1 - k0 + 1;
            off[m] = used;
            used += len[m];
        }
    }
};
template <int NM>
struct Mel {
    static constexpr MelShape<NM> shape{};
};

// 8-point DFT of u[n] = (w[n].x x[n].x, w[n].y x[n].y), the window folded into the first
// radix-2 layer (n, n + 4).  Even outputs are the 4-point DFT of the sums, odd outputs the
// 4-point DFT of the differences times W8^n.
__device__ __forceinline__ void dft8_windowed(const float2 (&x)[8], const float2 *w, float2 (&X)[8]) {
    float2 s[4], d[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 wa = w[j], wb = w[j + 4];
        const float ar = wa.x * x[j].x, ai = wa.y * x[j].y;
        s[j] = make_float2(fmaf(wb.x, x[j + 4].x, ar), fmaf(wb.y, x[j + 4].y, ai));
        d[j] = make_float2(fmaf(-wb.x, x[j + 4].x, ar), fmaf(-wb.y, x[j + 4].y, ai));
    }
    const float h = 0.70710678118654752f;
    {
        const float2 p = make_float2(s[0].x + s[2].x, s[0].y + s[2].y), q = make_float2(s[0].x - s[2].x, s[0].y - s[2].y);
        const float2 r = make_float2(s[1].x + s[3].x, s[1].y + s[3].y), t = make_float2(s[1].x - s[3].x, s[1].y - s[3].y);
        X[0] = make_float2(p.x + r.x, p.y + r.y);
        X[4] = make_float2(p.x - r.x, p.y - r.y);
        X[2] = make_float2(q.x + t.y, q.y - t.x);   // q - i t
        X[6] = make_float2(q.x - t.y, q.y + t.x);   // q + i t
    }
    {
        const float2 e1 = make_float2(h * (d[1].x + d[1].y), h * (d[1].y - d[1].x));    // W8 d1
        const float2 e2 = make_float2(d[2].y, -d[2].x);                                // W8^2 d2
        const float2 e3 = make_float2(h * (d[3].y - d[3].x), -h * (d[3].x + d[3].y));   // W8^3 d3
        const float2 p = make_float2(d[0].x + e2.x, d[0].y + e2.y), q = make_float2(d[0].x - e2.x, d[0].y - e2.y);
        const float2 r = make_float2(e1.x + e3.x, e1.y + e3.y), t = make_float2(e1.x - e3.x, e1.y - e3.y);
        X[1] = make_float2(p.x + r.x, p.y + r.y);
        X[5] = make_float2(p.x - r.x, p.y - r.y);
        X[3] = make_float2(q.x + t.y, q.y - t.x);
        X[7] = make_float2(q.x - t.y, q.y + t.x);
    }
}

// 5-point DFT in place, W5 = exp(-2 pi i / 5), with t1 = y1 + y4, t2 = y2 + y3,
// t3 = y1 - y4, t4 = y2 - y3:
//   Y0 = y0 + t1 + t2,
//   Y1, Y4 = y0 + c1 t1 + c2 t2 -/+ i (s1 t3 + s2 t4),
//   Y2, Y3 = y0 + c2 t1 + c1 t2 -/+ i (s2 t3 - s1 t4),
// c1, s1 = cos, sin (2 pi / 5) and c2, s2 = cos, sin (4 pi / 5).  Each complex value is one
// packed (re, im) pair: complex sums and real scalings are single f32x2 instructions, and
// -/+ i u is the swapped pair times (1, -1) or (-1, 1).
__device__ __forceinline__ float2 p_add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 p_mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 p_fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ void dft5p(float2 &y0, float2 &y1, float2 &y2, float2 &y3, float2 &y4) {
    const float c1 = 0.30901699437494745f, c2 = -0.80901699437494734f;
    const float s1 = 0.95105651629515353f, s2 = 0.58778525229247325f;
    const float2 C1 = make_float2(c1, c1), C2 = make_float2(c2, c2);
    const float2 S1 = make_float2(s1, s1), S2 = make_float2(s2, s2), NS1 = make_float2(-s1, -s1);
    const float2 M1 = make_float2(-1.0f, -1.0f), PM = make_float2(1.0f, -1.0f), MP = make_float2(-1.0f, 1.0f);
    const float2 t1 = p_add(y1, y4), t2 = p_add(y2, y3);
    const float2 t3 = p_fma(M1, y4, y1), t4 = p_fma(M1, y3, y2);
    const float2 a = p_fma(C2, t2, p_fma(C1, t1, y0));
    const float2 c = p_fma(C1, t2, p_fma(C2, t1, y0));
    const float2 u = p_fma(S2, t4, p_mul(S1, t3));
    const float2 v = p_fma(NS1, t4, p_mul(S2, t3));
    y0 = p_add(y0, p_add(t1, t2));
    const float2 us = make_float2(u.y, u.x), vs = make_float2(v.y, v.x);
    y1 = p_fma(PM, us, a);   // a - i u
    y4 = p_fma(MP, us, a);   // a + i u
    y2 = p_fma(PM, vs, c);
    y3 = p_fma(MP, vs, c);
}

// 25-point DFT in place, n = 5 a + b, k = c + 5 e: 5-point DFTs over a (for each b), the
// twiddles W25^(b c), 5-point DFTs over b (for each c).  On return v[5 c + e] = X[c + 5 e].
__device__ __forceinline__ void dft25(float2 (&v)[25]) {
    // (cos, sin)(2 pi j / 25), j = 1 .. 16
    constexpr float C[16] = {0.96858316112863108f, 0.87630668004386358f, 0.72896862742141155f,
                             0.53582679497899655f, 0.30901699437494745f, 0.062790519529313527f,
                             -0.1873813145857246f, -0.42577929156507272f, -0.63742398974868975f,
                             -0.80901699437494734f, -0.92977648588825135f, -0.99211470131447776f,
                             -0.99211470131447788f, -0.92977648588825146f, -0.80901699437494778f,
                             -0.63742398974868952f};
    constexpr float S[16] = {0.24868988716485479f, 0.48175367410171532f, 0.68454710592868862f,
                             0.84432792550201508f, 0.95105651629515353f, 0.99802672842827156f,
                             0.98228725072868872f, 0.90482705246601947f, 0.77051324277578925f,
                             0.58778525229247325f, 0.36812455268467814f, 0.12533323356430454f,
                             -0.12533323356430429f, -0.36812455268467792f, -0.58778525229247269f,
                             -0.77051324277578936f};
#pragma unroll
    for (int b = 0; b < 5; ++b) dft5p(v[b], v[5 + b], v[10 + b], v[15 + b], v[20 + b]);
    // now v[5 c + b] = U[b][c]; multiply by W25^(b c) = (cos, -sin)(2 pi b c / 25)
#pragma unroll
    for (int b = 1; b < 5; ++b)
#pragma unroll
        for (int c = 1; c < 5; ++c) {
            const float cs = C[b * c - 1], sn = S[b * c - 1];
            const float2 a = v[5 * c + b];
            v[5 * c + b] = make_float2(a.x * cs + a.y * sn, a.y * cs - a.x * sn);
        }
#pragma unroll
    for (int c = 0; c < 5; ++c) dft5p(v[5 * c], v[5 * c + 1], v[5 * c + 2], v[5 * c + 3], v[5 * c + 4]);
}

// Order-preserving map float -> uint32 (for atomicMax over signed floats).
__device__ __forceinline__ uint32_t f2key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Stage A: frame = lane, n2 = warp, warp + 8, ...: the 8-point DFT over n1 of the windowed
// z[(25 n1 + 8 n2) mod 200], stored at [k1][n2][frame].  The window pairs and gather offsets
// of each n2 come from a small table in shared memory (one broadcast read per value).
__device__ __forceinline__ void dft8_item(const float *__restrict__ xf, const ARow *__restrict__ r,
                                          float2 *__restrict__ dst) {
    float2 u[8], y[8], w[8];
#pragma unroll
    for (int n1 = 0; n1 < 8; ++n1) {
        w[n1] = r->w[n1];
        u[n1] = *reinterpret_cast<const float2 *>(xf + r->off[n1]);
    }
    dft8_windowed(u, w, y);
#pragma unroll
    for (int k1 = 0; k1 < 8; ++k1) dst[k1 * N2 * TF] = y[k1];
}
__device__ __forceinline__ void stage_a(const float *__restrict__ xf, const ARow *__restrict__ at,
                                        float2 *__restrict__ R2, int warp, int lane) {
    for (int n2 = warp; n2 < N2; n2 += NWARP) dft8_item(xf, at + n2, R2 + n2 * TF + lane);
}

// Stage C: frame = lane, bin pairs (k, 200 - k) with k = warp + 8 i in 1 .. 100.  Z[k] sits at
// [k mod 8][k mod 25].  With A = Z[k], B = Z[200 - k]: 2E = A + conj B, 2O = -i (A - conj B),
// X[k] = E + W400^k O, X[200 - k] = conj(E - W400^k O).  The powers are kept x 4 (c_mel_w
// carries the 1/4); bins 0 and 200 are not stored.
__device__ __forceinline__ void stage_c(const float2 *__restrict__ R2, float *__restrict__ P, int warp, int lane) {
    const float2 *za = R2 + warp * N2 * TF + lane;                  // k mod 8 = warp
    const float2 *zb = R2 + ((8 - warp) & 7) * N2 * TF + lane;      // (200 - k) mod 8
    int k = warp == 0 ? NWARP : warp;
    int ka = k % 25;                                                // k mod 25
#pragma unroll 4
    for (; k <= 100; k += NWARP) {
        const int kb = ka == 0 ? 0 : 25 - ka;                       // (200 - k) mod 25
        const float2 A = za[ka * TF];
        const float2 B = zb[kb * TF];
        const float er = A.x + B.x, ei = A.y - B.y;
        const float o_r = A.y + B.y, o_i = B.x - A.x;
        const float2 w = c_tw[k];
        const float vr = w.x * o_r - w.y * o_i, vi = w.x * o_i + w.y * o_r;
        const float pr = er + vr, pi = ei + vi, mr = er - vr, mi = ei - vi;
        P[(k - 1) * TF + lane] = pr * pr + pi * pi;
        P[(199 - k) * TF + lane] = mr * mr + mi * mi;   // bin 200 - k
        ka = ka + 8 >= 25 ? ka + 8 - 25 : ka + 8;
    }
}

// Stage D for warp W: frame = lane, filters m = W + 8 j: the sparse projection (straight-line:
// bins and weight offsets are compile-time), log10 with floor 1e-10, into the log-mel tile
// [frame][m]; the running maximum over valid frames.
template <int NM, int W, int J>
__device__ __forceinline__ void stage_d(const float *__restrict__ P, float *__restrict__ Mt, int lane, bool valid,
                                        float &lmax) {
    constexpr int m = W + NWARP * J;
    if constexpr (m < NM) {
        constexpr int T = NM == 128 ? 1 : 0;
        constexpr int k0 = Mel<NM>::shape.start[m] - 1, len = Mel<NM>::shape.len[m], off = Mel<NM>::shape.off[m];
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < len; ++i) acc = fmaf(c_mel_w[T][off + i], P[(k0 + i) * TF + lane], acc);
        // log10 via the hardware log2 (log10 x = log2 x * log10 2); at the floor exactly -10.
        float lg2;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg2) : "f"(acc));
        const float lg = acc > 1e-10f ? lg2 * 0.30102999566398120f : -10.0f;
        Mt[lane * MT_STRIDE + m] = lg;
        lmax = fmaxf(lmax, valid ? lg : -INFINITY);
        stage_d<NM, W, J + 1>(P, Mt, lane, valid, lmax);
    }
}

#define WH_WARP_SWITCH(call_w)                                                                       \
    switch (warp) {                                                                                  \
        case 0: call_w(0); break;                                                                    \
        case 1: call_w(1); break;                                                                    \
        case 2: call_w(2); break;                                                                    \
        case 3: call_w(3); break;                                                                    \
        case 4: call_w(4); break;                                                                    \
        case 5: call_w(5); break;                                                                    \
        case 6: call_w(6); break;                                                                    \
        default: call_w(7); break;                                                                   \
    }

// Window b starts at pcm + b * stride and holds min(n, total - b * stride) samples (a batch of
// clips: stride = n, total = batch * n; one long clip cut into 30-s windows: stride = n =
// 480000, total = the clip's length).
struct Tile {
    const float *x;   // the window's first sample
    long long n;      // samples the window holds
    long long s0;     // span start (160 t0 - 200)
    int b, t0, nf;
    bool fast;        // the span lies inside the clip and is 16-byte aligned
};
__device__ __forceinline__ Tile tile_of(int t, const float *pcm, long long n, long long stride, long long total) {
    Tile T;
    T.b = t / TILES;
    T.t0 = (t - T.b * TILES) * TF;
    T.nf = min(TF, N_FRAMES - T.t0);
    T.x = pcm + (long long)T.b * stride;
    T.n = min(n, total - (long long)T.b * stride);
    T.s0 = (long long)HOP * T.t0 - N_FFT / 2;
    const long long lim = T.n < N_SAMPLES ? T.n : N_SAMPLES;
    T.fast = T.s0 >= 0 && T.s0 + SPAN <= lim && ((reinterpret_cast<uintptr_t>(T.x + T.s0) & 15) == 0);
    return T;
}

// One persistent grid (all blocks resident: a cooperative launch) walks the tiles of every
// window; each block prefetches its next tile's samples into registers while it finishes the
// current one.  Every tile writes its log10 values and raises its window's maximum; after a
// grid-wide barrier all blocks apply the clamp (max(x, g - 8) + 4) / 4 to an equal share of
// the output.  ws holds the batch's window maxima (order-preserving keys) then the barrier's
// arrival count, all zero at launch.
template <int NM>
__global__ void __launch_bounds__(THREADS, 2) k_logmel(const float *__restrict__ pcm, long long n, long long stride,
                                                       long long total, int batch, float *__restrict__ mel,
                                                       uint32_t *__restrict__ ws, DevCtl ctl) {
    extern __shared__ float4 smem4[];
    float *R1 = reinterpret_cast<float *>(smem4);             // staged samples, then the power [bin - 1][frame]
    float2 *R2 = reinterpret_cast<float2 *>(R1 + R1_FLOATS);  // spectra [k1][k2][frame], then the log-mel tile
    __shared__ float red[NWARP];
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tiles = TILES * batch;
    float4 pf[PF];   // the next tile's samples (fast tiles only)
    bool have_pf = false;

    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        // The stage-A table (window pairs and gather offsets per n2) goes into the slack above
        // the staged samples; then the samples 160 t0 - 200 ... (pad/truncate to 480000, then
        // reflect by 200), from the prefetch registers or straight from global memory.
        {
            const int4 *src = reinterpret_cast<const int4 *>(c_arow);
            int4 *dst = reinterpret_cast<int4 *>(R1 + A_TABLE);
            for (int i = tid; i < (int)(sizeof(c_arow) / 16); i += THREADS) dst[i] = src[i];
        }
        if (have_pf) {
#pragma unroll
            for (int u = 0; u < PF; ++u) {
                const int q = tid + u * THREADS;
                if (q < SPAN / 4) {
                    float *d = R1 + seg_pos(4 * q);   // the four samples share a row (160 % 4 == 0)
                    *reinterpret_cast<float2 *>(d) = make_float2(pf[u].x, pf[u].y);
                    *reinterpret_cast<float2 *>(d + 2) = make_float2(pf[u].z, pf[u].w);
                }
            }
        } else {
            const Tile T = tile_of(t, pcm, n, stride, total);
            if (T.fast) {
                const float4 *src = reinterpret_cast<const float4 *>(T.x + T.s0);
                for (int q = tid; q < SPAN / 4; q += THREADS) {
                    const float4 v = __ldg(src + q);
                    float *d = R1 + seg_pos(4 * q);
                    *reinterpret_cast<float2 *>(d) = make_float2(v.x, v.y);
                    *reinterpret_cast<float2 *>(d + 2) = make_float2(v.z, v.w);
                }
            } else {
                for (int j = tid; j < SPAN; j += THREADS) {
                    long long si = T.s0 + j;
                    si = si < 0 ? -si : si;
                    si = si > N_SAMPLES - 1 ? 2LL * (N_SAMPLES - 1) - si : si;
                    R1[seg_pos(j)] = (si < T.n) ? __ldg(T.x + si) : 0.0f;
                }
            }
        }
        __syncthreads();

        stage_a(R1 + ROW * lane, reinterpret_cast<const ARow *>(R1 + A_TABLE), R2, warp, lane);
        __syncthreads();

        // Stage B: frame = lane, k1 = warp: the 25-point DFT over n2, in place;
        // [k1][k2][frame] then holds Z[(25 k1 + 176 k2) mod 200].
        {
            float2 *col = R2 + warp * N2 * TF + lane;
            float2 v[25];
#pragma unroll
            for (int i = 0; i < 25; ++i) v[i] = col[i * TF];
            dft25(v);
#pragma unroll
            for (int c = 0; c < 5; ++c)
#pragma unroll
                for (int e = 0; e < 5; ++e) col[(c + 5 * e) * TF] = v[5 * c + e];
        }
        __syncthreads();

        // Prefetch the next tile's samples (the loads complete behind stages C and D).
        {
            const int tn = t + gridDim.x;
            have_pf = false;
            if (tn < tiles) {
                const Tile N = tile_of(tn, pcm, n, stride, total);
                if (N.fast) {
                    const float4 *src = reinterpret_cast<const float4 *>(N.x + N.s0);
#pragma unroll
                    for (int u = 0; u < PF; ++u) {
                        const int q = tid + u * THREADS;
                        if (q < SPAN / 4) pf[u] = __ldg(src + q);
                    }
                    have_pf = true;
                }
            }
        }

        float *P = R1;
        stage_c(R2, P, warp, lane);
        __syncthreads();

        const int tb = t / TILES, t0 = (t - tb * TILES) * TF, nf = min(TF, N_FRAMES - t0);
        float lmax = -INFINITY;
        float *Mt = reinterpret_cast<float *>(R2);
        const bool valid = lane < nf;
#define WH_STAGE_D(w) stage_d<NM, w, 0>(P, Mt, lane, valid, lmax)
        WH_WARP_SWITCH(WH_STAGE_D)
#undef WH_STAGE_D
        __syncthreads();

        // Frame-major store of the log10 values: one row of NM per frame, lanes over m.
        float *out = mel + ((long long)tb * N_FRAMES + t0) * NM;
#pragma unroll
        for (int f = warp; f < TF; f += NWARP) {
            if (f >= nf) break;
#pragma unroll
            for (int m0 = 0; m0 < NM; m0 += 32)
                if (m0 + lane < NM) out[(long long)f * NM + m0 + lane] = Mt[f * MT_STRIDE + m0 + lane];
        }
        lmax = warp_max(lmax);
        if (lane == 0) red[warp] = lmax;
        __syncthreads();   // also: this tile's shared-memory reads are done before the next staging
        if (tid < 32) {
            float v = tid < NWARP ? red[tid] : -INFINITY;
            v = warp_max(v);
            if (tid == 0) atomicMax(ws + tb, f2key(v));
        }
    }

    // Grid-wide barrier: every tile's values and maxima are written.  Bounded: on expiry the
    // status word records WH_ETIMEOUT and the block returns without clamping.
    __syncthreads();
    if (tid == 0) {
        int ok = 1;
        __threadfence();
        atomicAdd(ws + batch, 1u);
        const uint64_t t_start = globaltimer_ns();
        for (uint32_t it = 0;; ++it) {
            uint32_t arrived;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(arrived) : "l"(ws + batch) : "memory");
            if (arrived >= gridDim.x) break;
            if ((it & 63u) == 63u && globaltimer_ns() - t_start > ctl.wait_ns) {
                set_status(ctl, WH_ETIMEOUT);
                ok = 0;
                break;
            }
        }
        abort_flag = !ok;
    }
    __syncthreads();
    if (abort_flag) return;

    // Clamp, an equal share per block: mel = (max(mel, g_b - 8) + 4) / 4, g_b window b's maximum.
    // A share may cover any number of windows (it is longer than a window once the batch has
    // more windows than the grid has blocks).  A thread's indices only grow, so each thread
    // follows the window its current index lies in and reloads the floor when it crosses
    // into the next one; eight float4 per thread are in flight at a time.
    constexpr int PER_WINDOW4 = N_FRAMES * NM / 4;
    constexpr int CU = 8;
    const long long all4 = (long long)batch * PER_WINDOW4;
    const long long chunk = (all4 + gridDim.x - 1) / gridDim.x;
    const long long lo = (long long)blockIdx.x * chunk, hi = min(all4, lo + chunk);
    if (lo >= hi) return;
    int b_cur = (int)((lo + tid) / PER_WINDOW4);
    long long next = (long long)(b_cur + 1) * PER_WINDOW4;   // first index of window b_cur + 1
    float fl = key2f(__ldcg(ws + min(b_cur, batch - 1))) - 8.0f;
    float4 *m4 = reinterpret_cast<float4 *>(mel);
    for (long long base = lo + tid; base < hi; base += CU * THREADS) {
        float4 v[CU];
#pragma unroll
        for (int u = 0; u < CU; ++u)
            if (base + u * THREADS < hi) v[u] = __ldcg(m4 + base + u * THREADS);
#pragma unroll
        for (int u = 0; u < CU; ++u) {
            const long long i = base + u * THREADS;
            if (i < hi) {
                if (i >= next) {   // i < all4, so the window index stays below batch
                    b_cur = (int)(i / PER_WINDOW4);
                    next = (long long)(b_cur + 1) * PER_WINDOW4;
                    fl = key2f(__ldcg(ws + b_cur)) - 8.0f;
                }
                float4 w = v[u];
                w.x = (fmaxf(w.x, fl) + 4.0f) * 0.25f;
                w.y = (fmaxf(w.y, fl) + 4.0f) * 0.25f;
                w.z = (fmaxf(w.z, fl) + 4.0f) * 0.25f;
                w.w = (fmaxf(w.w, fl) + 4.0f) * 0.25f;
                m4[i] = w;
            }
        }
    }
}
#undef WH_WARP_SWITCH

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
    const double pi = 3.14159265358979323846;
    double hann[N_FFT];
    for (int j = 0; j < N_FFT; ++j) hann[j] = 0.5 - 0.5 * std::cos(2.0 * pi * j / N_FFT);
    ARow arow[N2];
    for (int n2 = 0; n2 < N2; ++n2)
        for (int n1 = 0; n1 < N1; ++n1) {
            const int m = (25 * n1 + 8 * n2) % 200;
            arow[n2].w[n1] = make_float2((float)hann[2 * m], (float)hann[2 * m + 1]);
            arow[n2].off[n1] = a_off(n1, n2);
        }
    float2 tw[101];
    for (int k = 0; k <= 100; ++k)
        tw[k] = make_float2((float)std::cos(2.0 * pi * k / N_FFT), (float)-std::sin(2.0 * pi * k / N_FFT));
    static MelTable mt[2];
    static std::once_flag once;
    static int build_rc = WH_OK;
    std::call_once(once, [] {
        build_rc = build_mel(80, mt[0]);
        if (build_rc == WH_OK) build_rc = build_mel(128, mt[1]);
    });
    if (build_rc != WH_OK) return build_rc;
    float w[2][MAXW];
    for (int t = 0; t < 2; ++t) {
        // The kernel stores the power of bins 1 .. 199 only and unrolls each filter over the
        // bins its compile-time shape names: both must hold for the table built here.
        const int nm = t ? 128 : 80;
        for (int m = 0; m < nm; ++m) {
            const int start = mt[t].start[m], len = mt[t].len[m], off = mt[t].off[m];
            if (start < 1 || start + len - 1 > N_BINS - 2) return WH_EINVAL;
            const int cs = t ? Mel<128>::shape.start[m] : Mel<80>::shape.start[m];
            const int cl = t ? Mel<128>::shape.len[m] : Mel<80>::shape.len[m];
            const int co = t ? Mel<128>::shape.off[m] : Mel<80>::shape.off[m];
            if (cs != start || cl != len || co != off) return WH_EINVAL;
        }
        for (int i = 0; i < MAXW; ++i) w[t][i] = 0.25f * mt[t].w[i];
    }
    if (cudaMemcpyToSymbol(c_arow, arow, sizeof(arow)) != cudaSuccess ||
        cudaMemcpyToSymbol(c_tw, tw, sizeof(tw)) != cudaSuccess ||
        cudaMemcpyToSymbol(c_mel_w, w, sizeof(w)) != cudaSuccess)
        return WH_ECUDA;
    if (cudaFuncSetAttribute(k_logmel<80>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(k_logmel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) != cudaSuccess)
        return WH_ECUDA;
    return WH_OK;
}

int frontend_launch(const float *pcm, int64_t n, int64_t stride, int64_t total, int batch, int n_mels, float *mel,
                    uint32_t *ws, const DevCtl &ctl, int num_sms, cudaStream_t s) {
    // window maxima and the barrier's arrival count start at zero
    if (cudaMemsetAsync(ws, 0, sizeof(uint32_t) * ((size_t)batch + 1), s) != cudaSuccess) return WH_ECUDA;
    const void *fn = n_mels == 128 ? reinterpret_cast<const void *>(k_logmel<128>)
                                   : reinterpret_cast<const void *>(k_logmel<80>);
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, THREADS, SMEM) != cudaSuccess || per_sm < 1)
        return WH_ECUDA;
    const long long tiles = (long long)TILES * batch;
    const long long resident = (long long)per_sm * num_sms;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)(tiles < resident ? tiles : resident));
    lc.blockDim = dim3(THREADS);
    lc.dynamicSmemBytes = SMEM;
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every block resident: the grid barrier
    attr[0].val.cooperative = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const long long nn = n, st = stride, tot = total;
    const cudaError_t e = n_mels == 128 ? cudaLaunchKernelEx(&lc, k_logmel<128>, pcm, nn, st, tot, batch, mel, ws, ctl)
                                        : cudaLaunchKernelEx(&lc, k_logmel<80>, pcm, nn, st, tot, batch, mel, ws, ctl);
    count_launch(1);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? WH_OK : WH_ECUDA;
}

}  // namespace wh
