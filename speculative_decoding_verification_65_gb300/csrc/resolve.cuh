// resolve.cuh -- exact inverse-CDF draws for the few rows whose fp32 draw
// lands near a cell boundary.
//
// The draw (P1 "The Algorithm, Step by Step", "Stop at the first rejection"
// and "Bonus token"; P2 "The correction that keeps the target in charge", the
// residual r(x) = norm(max(0, p(x) - q(x)))) takes the smallest x with
// C(x) > u * R, C the running sum of the weights and R their total.  The fp32
// kernels compute C to about 1e-6 of R; where u * R lies closer than a guard
// to the edges of the cell they chose, the row is listed and drawn again here
// with arithmetic accurate to about 1e-12 of R.  Only fp32 and integer
// instructions are used (this GPU's fp64 pipe is narrow):
//
//   * every weight e = 2^((x - m) * log2(e) / T) is computed in float-float
//     arithmetic (the exponent as a pair of floats, a 256-entry table of
//     2^(i/256) as float pairs, a degree-4 series on the remaining
//     |a| <= ln2/512; about 4e-13 relative error), then rounded to a 64-bit
//     fixed-point integer E in units of 2^-51 of the row maximum's weight;
//   * sums of those integers are exact, so they depend neither on the order
//     nor on which CTA added them;
//   * a residual weight is proportional to max(0, E_t(x) Z_d - E_d(x) Z_t),
//     Z the rows' masses (p = E_t / Z_t, q = E_d / Z_d).  One pass sorts each
//     element by the sign of that difference using the fp32 masses (checked
//     afterwards to agree with the exact ratio within 2^-16): clearly
//     positive elements add E_t and E_d to their chunk's sums A_t and A_d,
//     clearly negative ones add nothing, and the rare elements within 2^-14
//     of the cut are listed and weighed once Z_t and Z_d are known.  A
//     chunk's residual mass is then Z_d A_t - Z_t A_d, a 128-bit integer;
//   * the last CTA to finish a row's chunks forms the chunk masses, their
//     prefix, the crossing chunk, and in it the crossing element, comparing
//     integers with floor(u * R) (exact for an integer running sum).
#pragma once

#include "device_common.cuh"
#include "exp2_table.h"

namespace spec_dev {

constexpr int RCH = 2048;            // elements per chunk (one work item)
constexpr int RTH = 256;             // threads of a resolving CTA
constexpr int RPT = RCH / RTH;       // elements per thread in a chunk
constexpr int RKCAP = 64;            // groups of undecided elements listed per row
constexpr int RKG = 32;              // groups a CTA collects in one chunk
constexpr int FIXB = 51;             // fixed-point weights in units of 2^-51
constexpr int RSHIFT = 40;           // residual products are kept in units of 2^40
constexpr int RMAXC = SPEC_MAX_V / RCH;
static_assert(RPT == 8, "a chunk gives each thread 8 elements");
static_assert(RKG <= RTH, "one thread per group of a chunk");
static_assert((long long)RCH << FIXB <= (1ll << 62), "chunk sums fit a signed 64-bit integer");

constexpr float LN2_HI = 0x1.62e430p-1f;     // ln 2 = LN2_HI + LN2_LO to ~2^-54
constexpr float LN2_LO = -0x1.05c610p-29f;
constexpr float LOG2E_HI = 0x1.715476p+0f;   // log2(e) = LOG2E_HI + LOG2E_LO to ~2^-51
constexpr float LOG2E_LO = 0x1.4ae0c0p-26f;
constexpr float RKAPPA = 0x1p-18f;           // undecided band of p/q around 1
constexpr float RRATIO_TOL = 0x1p-19f;       // required agreement of the fp32 and exact mass ratios

enum { RJ_RESIDUAL = 1, RJ_TARGET = 2 };

typedef __int128 i128;
typedef unsigned __int128 u128;

// One draw to resolve.  RJ_TARGET: weights 2^((x - mt) * c) of the target
// row alone (a bonus or a sampled row); RJ_RESIDUAL: both rows.
struct alignas(16) RJob {
    const void *t_arr, *d_arr;
    long long t_row, d_row;
    int mode;
    float mt, md;    // row maxima (of the kept sets, when filtered)
    float rzt, rzd;  // 1 / (fp32 masses): used only to sort elements by sign
    float ch, cl;    // log2(e) / T as a float pair
    float u;
    int filt;        // top-k / top-p: x counts in a row iff key > k_ or (key == k_ and x <= i_)
    unsigned int kt, kd;
    int it, id;
    int b;           // the trace row (spec_verify_trace), or unused
    long long out_pos;  // where the token goes in the output array
};
static_assert(sizeof(RJob) % 16 == 0, "an exact-draw record is whole 16-byte vectors");

// Per-chunk sums (fixed point, units of 2^-51 of each row's maximum weight):
// the positive set's A_t, A_d and every element's Z_t, Z_d.
struct alignas(32) RzRec {
    long long at, ad, zt, zd;
};

// A group of undecided elements of one chunk: elements whose logits differ
// by the same amount t(x) - d(x) have the same p/q, so one sign decides them
// all once the masses are known.
struct alignas(32) RkRec {
    long long et, ed;  // their fixed-point sums
    int chunk;
    int pad[3];
};

// Shared memory of a resolving CTA.
struct RSmem {
    RJob job;  // the current work item's draw
    float2 tab[256];
    long long red[RTH / 32][4];
    unsigned int gkey[RKG][2];        // undecided groups of the current chunk: t - d as a float pair
    unsigned long long gsum[RKG][2];
    int gcnt;
    long long next;
};

__device__ __forceinline__ i128 mk128(unsigned long long lo, unsigned long long hi)
{
    return (i128)(((u128)hi << 64) | (u128)lo);
}
__device__ __forceinline__ unsigned long long lo64(i128 v) { return (unsigned long long)(u128)v; }
__device__ __forceinline__ unsigned long long hi64(i128 v) { return (unsigned long long)((u128)v >> 64); }

__device__ __forceinline__ void load_exp2_table(float2 *tab)
{
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
        tab[i] = make_float2(kExp2Tab[i][0], kExp2Tab[i][1]);
}

// log2(e) / T as a pair of floats (about 2^-47 relative): the remainder of a
// correctly rounded quotient is exact, so LOG2E_HI - ch * T loses nothing.
__device__ __forceinline__ void exp_coef(float T, float &ch, float &cl)
{
    ch = __fdiv_rn(LOG2E_HI, T);
    const float rem = __fmaf_rn(-ch, T, LOG2E_HI);
    cl = __fdiv_rn(__fadd_rn(rem, LOG2E_LO), T);
}

// rh * 2^(n + 51) + rl * 2^(n + 51) rounded to an integer: rh's 24-bit
// significand shifted by n + 28 + (rh's exponent), right shifts rounding
// half up, plus rl * 2^(n + 51), which is below 2^30 in magnitude.
__device__ __forceinline__ long long fix_of(float rh, float rl, int n)
{
    const unsigned int rb = __float_as_uint(rh);
    const unsigned long long M = (unsigned long long)((rb & 0x7fffffu) | 0x800000u);
    const int s = n + FIXB - 150 + (int)(rb >> 23);
    const unsigned long long hi =
        (s >= 0) ? (M << s) : ((s > -40) ? ((M + (1ull << (-s - 1))) >> (-s)) : 0ull);
    const int lo = __float2int_rn(__fmul_rn(rl, __int_as_float((n + FIXB + 127) << 23)));
    return (long long)hi + (long long)lo;
}

// ---- weights two at a time, in packed f32x2 arithmetic (each half rounds
// exactly like the scalar instruction)

__device__ __forceinline__ unsigned long long fx2(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void ux2(unsigned long long v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long addx2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long subx2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long mulx2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long fmax2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// e = 2^((x - m) * c) as an integer in units of 2^-51 (x <= m, so e <= 1),
// rounded to nearest, for two elements at once: x0 against maximum m0 and x1
// against m1, the same coefficient c = ch + cl.  0 when the exponent is below
// -60 (e < 2^-60, under 2^-9 of a unit), x is -inf, or ok0 / ok1 is false
// (masked or absent elements).  a0 / a1 receive e as floats (without the
// 2^51 scale) for sign decisions.  Every operation an exact split relies on
// is an explicitly rounded instruction, which the compiler does not fuse.
__device__ __forceinline__ void efix2(float x0, float x1, float m0, float m1, bool ok0, bool ok1,
                                      float ch, float cl, const float2 *tab, long long &E0,
                                      long long &E1, float &a0, float &a1)
{
    const unsigned long long X = fx2(x0, x1), Mx = fx2(m0, m1), NMx = fx2(-m0, -m1);
    const unsigned long long C = fx2(ch, ch), NC = fx2(-ch, -ch), CL = fx2(cl, cl);
    const unsigned long long DH = subx2(X, Mx);
    const unsigned long long SH = mulx2(DH, C), NSH = mulx2(DH, NC);
    float sh0, sh1;
    ux2(SH, sh0, sh1);
    ok0 = ok0 && (sh0 >= -60.0f);  // also -inf and NaN
    ok1 = ok1 && (sh1 >= -60.0f);
    const unsigned long long BB = subx2(DH, X);
    const unsigned long long DL = addx2(subx2(X, subx2(DH, BB)), subx2(NMx, BB));
    const unsigned long long SL = addx2(fmax2(DH, C, NSH), fmax2(DH, CL, mulx2(DL, C)));
    const unsigned long long T = mulx2(SH, fx2(256.0f, 256.0f));
    const unsigned long long MG = fx2(0x1.8p23f, 0x1.8p23f);
    const unsigned long long TM = addx2(T, MG);
    float tm0, tm1;
    ux2(TM, tm0, tm1);
    const int j0 = ok0 ? __float_as_int(tm0) - 0x4b400000 : 0;
    const int j1 = ok1 ? __float_as_int(tm1) - 0x4b400000 : 0;
    const unsigned long long JF = subx2(TM, MG);
    const unsigned long long F = mulx2(subx2(T, JF), fx2(0x1p-8f, 0x1p-8f));
    const unsigned long long GH = addx2(F, SL);
    const unsigned long long GB = subx2(GH, F);
    const unsigned long long GL = addx2(subx2(F, subx2(GH, GB)), subx2(SL, GB));
    const unsigned long long L2H = fx2(LN2_HI, LN2_HI);
    const unsigned long long AH = mulx2(GH, L2H), NAH = mulx2(GH, fx2(-LN2_HI, -LN2_HI));
    const unsigned long long AL =
        addx2(fmax2(GH, L2H, NAH), fmax2(GH, fx2(LN2_LO, LN2_LO), mulx2(GL, L2H)));
    unsigned long long Pp = fmax2(AH, fx2(1.0f / 24.0f, 1.0f / 24.0f), fx2(1.0f / 6.0f, 1.0f / 6.0f));
    Pp = fmax2(AH, Pp, fx2(0.5f, 0.5f));
    Pp = mulx2(mulx2(AH, AH), Pp);
    const unsigned long long ML = addx2(AL, fmax2(AH, AL, Pp));
    const float2 T0 = tab[j0 & 255], T1 = tab[j1 & 255];
    const unsigned long long TX = fx2(T0.x, T1.x), TY = fx2(T0.y, T1.y);
    const unsigned long long PH = mulx2(TX, AH);
    const unsigned long long PL = fmax2(TX, AH, mulx2(TX, NAH));
    const unsigned long long REST = addx2(PL, fmax2(TX, ML, fmax2(TY, AH, TY)));
    const unsigned long long RH = addx2(TX, PH);
    const unsigned long long RL = addx2(subx2(PH, subx2(RH, TX)), REST);
    float rh0, rh1, rl0, rl1;
    ux2(RH, rh0, rh1);
    ux2(RL, rl0, rl1);
    const int n0 = j0 >> 8, n1 = j1 >> 8;
    a0 = ok0 ? __fmul_rn(rh0, __int_as_float((n0 + 127) << 23)) : 0.0f;
    a1 = ok1 ? __fmul_rn(rh1, __int_as_float((n1 + 127) << 23)) : 0.0f;
    E0 = ok0 ? fix_of(rh0, rl0, n0) : 0;
    E1 = ok1 ? fix_of(rh1, rl1, n1) : 0;
}

// Whether element x of a row counts (top-k / top-p kept set); always when
// the job is unfiltered.  The key is the float's bits mapped to an unsigned
// order (a bf16 value keeps its 16 significant bits).
template <int DT>
__device__ __forceinline__ bool rj_kept(const RJob &J, float v, int x, bool draft)
{
    if (!J.filt)
        return true;
    const unsigned int bits = __float_as_uint(v);
    const unsigned int key = ((bits & 0x80000000u) ? ~bits : (bits | 0x80000000u)) &
                             ((DT == SPEC_BF16) ? 0xffff0000u : 0xffffffffu);
    const unsigned int kap = draft ? J.kd : J.kt;
    const int iota = draft ? J.id : J.it;
    return key > kap || (key == kap && x <= iota);
}

__device__ __forceinline__ long long warp_sum_ll(long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One chunk (elements q*RCH .. q*RCH + RCH - 1) of a job: the CTA writes the
// chunk's record and appends its groups of undecided elements to `kinks`
// (the count in *kcnt may exceed RKCAP; the finishing step then does not use
// the list).  Thread t takes elements q*RCH + 8t .. 8t+7.
template <int DT>
__device__ void resolve_chunk(const RJob &J, int q, int V, RzRec *rec, RkRec *kinks,
                              unsigned int *kcnt, RSmem &S)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool residual = J.mode == RJ_RESIDUAL;
    if (tid < RKG) {
        S.gkey[tid][0] = S.gkey[tid][1] = 0xffffffffu;  // a NaN pair: matches no difference
        S.gsum[tid][0] = S.gsum[tid][1] = 0ull;
    }
    if (tid == 0)
        S.gcnt = 0;
    __syncthreads();
    using L = Lg<DT>;
    const int e0 = q * RCH + tid * RPT;
    // the record's fields once, in registers
    const float mt = J.mt, md = J.md, ch = J.ch, cl = J.cl, rzt = J.rzt, rzd = J.rzd;
    const bool filt = J.filt != 0;
    long long at = 0, ad = 0, zt = 0, zd = 0;
    bool overflow = false;
    // one 16-byte vector of each row at a time (fp32: two vectors, bf16: one)
#pragma unroll
    for (int h = 0; h < RPT / L::VEC; ++h) {
        const int v0 = e0 + h * L::VEC;
        const uint4 rt = row_vec<DT>(J.t_arr, (size_t)J.t_row, v0 / L::VEC, V);
        const uint4 rd = residual ? row_vec<DT>(J.d_arr, (size_t)J.d_row, v0 / L::VEC, V) : rt;
        float xt[L::VEC], xd[L::VEC];
        L::unpack(rt, xt);
        L::unpack(rd, xd);
        if (!residual) {
#pragma unroll
            for (int i = 0; i < L::VEC; i += 2) {
                long long E0, E1;
                float a0, a1;
                efix2(xt[i], xt[i + 1], mt, mt,
                      v0 + i < V && (!filt || rj_kept<DT>(J, xt[i], v0 + i, false)),
                      v0 + i + 1 < V && (!filt || rj_kept<DT>(J, xt[i + 1], v0 + i + 1, false)),
                      ch, cl, S.tab, E0, E1, a0, a1);
                zt += E0 + E1;
            }
            continue;
        }
#pragma unroll
        for (int i = 0; i < L::VEC; ++i) {
            const int x = v0 + i;
            long long Et, Ed;
            float ft, fd;
            efix2(xt[i], xd[i], mt, md, x < V && (!filt || rj_kept<DT>(J, xt[i], x, false)),
                  x < V && (!filt || rj_kept<DT>(J, xd[i], x, true)), ch, cl, S.tab, Et, Ed, ft, fd);
            zt += Et;
            zd += Ed;
            if (Et == 0 && Ed == 0)
                continue;
            const float Pp = ft * rzt, Qq = fd * rzd;
            if (Pp > Qq * (1.0f + RKAPPA)) {
                at += Et;
                ad += Ed;
            } else if (!(Qq > Pp * (1.0f + RKAPPA))) {
                // undecided: group it by t(x) - d(x), an exact float pair
                const float dh = __fsub_rn(xt[i], xd[i]);
                const float bb = __fsub_rn(dh, xt[i]);
                const float dl = __fadd_rn(__fsub_rn(xt[i], __fsub_rn(dh, bb)), __fsub_rn(-xd[i], bb));
                const unsigned int k0 = __float_as_uint(dh), k1 = __float_as_uint(dl);
                const int n = min(*reinterpret_cast<volatile int *>(&S.gcnt), RKG);
                int slot = -1;
                for (int g = 0; g < n; ++g)
                    if (S.gkey[g][0] == k0 && S.gkey[g][1] == k1) {
                        slot = g;
                        break;
                    }
                if (slot < 0) {
                    // a new group (two threads may both open one for the same
                    // difference; each group is weighed on its own, so that is harmless)
                    slot = atomicAdd(&S.gcnt, 1);
                    if (slot < RKG) {
                        S.gkey[slot][0] = k0;
                        S.gkey[slot][1] = k1;
                    }
                }
                if (slot < RKG) {
                    atomicAdd(&S.gsum[slot][0], (unsigned long long)Et);
                    atomicAdd(&S.gsum[slot][1], (unsigned long long)Ed);
                } else {
                    overflow = true;
                }
            }
        }
    }
    if (__syncthreads_or(overflow) && tid == 0)
        atomicAdd(kcnt, (unsigned int)RKCAP + 1u);  // too many groups: the finishing step's slow path
    // the chunk's groups go to the sequence's list
    const int ng = min(S.gcnt, RKG);
    if (tid < ng) {
        const unsigned int k = atomicAdd(kcnt, 1u);
        if (k < (unsigned int)RKCAP) {
            RkRec r;
            r.et = (long long)S.gsum[tid][0];
            r.ed = (long long)S.gsum[tid][1];
            r.chunk = q;
            r.pad[0] = r.pad[1] = r.pad[2] = 0;
            kinks[k] = r;
            __threadfence();
        }
    }
    at = warp_sum_ll(at);
    ad = warp_sum_ll(ad);
    zt = warp_sum_ll(zt);
    zd = warp_sum_ll(zd);
    if (lane == 0) {
        S.red[warp][0] = at;
        S.red[warp][1] = ad;
        S.red[warp][2] = zt;
        S.red[warp][3] = zd;
    }
    __syncthreads();
    if (tid == 0) {
        long long r0 = 0, r1 = 0, r2 = 0, r3 = 0;
        for (int w = 0; w < RTH / 32; ++w) {
            r0 += S.red[w][0];
            r1 += S.red[w][1];
            r2 += S.red[w][2];
            r3 += S.red[w][3];
        }
        __stcg(reinterpret_cast<longlong2 *>(rec), make_longlong2(r0, r1));
        __stcg(reinterpret_cast<longlong2 *>(rec) + 1, make_longlong2(r2, r3));
    }
}

// ------------------------------------------------------------ finishing
//
// One CTA of RFTH threads per listed row, after every chunk is done: the
// row's masses, the chunk masses, their prefix, the crossing chunk, and in
// it the crossing element.  Thread t holds chunk record t, and RFPT
// consecutive elements of the crossing chunk.

constexpr int RFTH = 512;
constexpr int RFPT = RCH / RFTH;
static_assert(RFTH >= RMAXC, "the finishing CTA holds one chunk record per thread");
static_assert(RFPT == 4, "the crossing chunk gives each finishing thread 4 elements");
static_assert(RKCAP <= RFTH, "one finishing thread per listed group");

struct RFSmem {
    float2 tab[256];
    unsigned long long zsum[RFTH / 32][4];
    unsigned long long wsum[RFTH / 32][2];
    unsigned long long W[RMAXC][2];   // chunk masses (i128 as lo, hi)
    int tok;
    int cstar;
    int lastp;
    int pad;
    unsigned long long before[2];
};

// Exclusive prefix of one i128 per thread in thread order; `total` gets the
// CTA's sum.  Called by every thread.
__device__ __forceinline__ i128 cta_excl_scan(i128 v, i128 &total, RFSmem &S)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    i128 x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long ylo = __shfl_up_sync(0xffffffffu, lo64(x), o);
        const unsigned long long yhi = __shfl_up_sync(0xffffffffu, hi64(x), o);
        if (lane >= o)
            x += mk128(ylo, yhi);
    }
    if (lane == 31) {
        S.wsum[warp][0] = lo64(x);
        S.wsum[warp][1] = hi64(x);
    }
    __syncthreads();
    i128 before = 0, tot = 0;
#pragma unroll 4
    for (int w = 0; w < RFTH / 32; ++w) {
        const i128 sw = mk128(S.wsum[w][0], S.wsum[w][1]);
        if (w < warp)
            before += sw;
        tot += sw;
    }
    total = tot;
    __syncthreads();
    return before + (x - v);
}

// Residual weight in the exact draw's units: max(0, E_t Z_d - E_d Z_t) / 2^40.
__device__ __forceinline__ i128 res_weight(long long Et, long long Ed, unsigned long long Zt,
                                           unsigned long long Zd)
{
    const i128 d = (i128)((u128)(unsigned long long)Et * Zd) -
                   (i128)((u128)(unsigned long long)Ed * Zt);
    return d > 0 ? (d >> RSHIFT) : (i128)0;
}

// Logits e0 .. e0+3 of a row (e0 a multiple of 4; -inf past V).
template <int DT>
__device__ __forceinline__ void rj_load4(const void *arr, long long row, int e0, int V,
                                         float (&x)[RFPT])
{
    using L = Lg<DT>;
    const uint4 r = row_vec<DT>(arr, (size_t)row, e0 / L::VEC, V);
    float y[L::VEC];
    L::unpack(r, y);
    const int o = e0 % L::VEC;
#pragma unroll
    for (int i = 0; i < RFPT; ++i)
        x[i] = y[(L::VEC == RFPT) ? i : (o + i) % L::VEC];
}

// Weights of elements e0 .. e0+3 in the exact draw: residual or E_t.
template <int DT>
__device__ __forceinline__ void rj_weights4(const RJob &J, int e0, int V, bool residual,
                                            unsigned long long Zt, unsigned long long Zd,
                                            i128 (&w)[RFPT], const float2 *tab)
{
    float xt[RFPT], xd[RFPT];
    rj_load4<DT>(J.t_arr, J.t_row, e0, V, xt);
    if (residual)
        rj_load4<DT>(J.d_arr, J.d_row, e0, V, xd);
    const bool filt = J.filt != 0;
    if (residual) {
#pragma unroll
        for (int i = 0; i < RFPT; ++i) {
            const int x = e0 + i;
            long long Et, Ed;
            float a0, a1;
            efix2(xt[i], xd[i], J.mt, J.md, x < V && (!filt || rj_kept<DT>(J, xt[i], x, false)),
                  x < V && (!filt || rj_kept<DT>(J, xd[i], x, true)), J.ch, J.cl, tab, Et, Ed, a0,
                  a1);
            w[i] = res_weight(Et, Ed, Zt, Zd);
        }
    } else {
#pragma unroll
        for (int i = 0; i < RFPT; i += 2) {
            const int x = e0 + i;
            long long E0, E1;
            float a0, a1;
            efix2(xt[i], xt[i + 1], J.mt, J.mt, x < V && (!filt || rj_kept<DT>(J, xt[i], x, false)),
                  x + 1 < V && (!filt || rj_kept<DT>(J, xt[i + 1], x + 1, false)), J.ch, J.cl, tab,
                  E0, E1, a0, a1);
            w[i] = (i128)E0;
            w[i + 1] = (i128)E1;
        }
    }
}

// floor(u * R) for u in [0, 1) (a float) and 0 <= R < 2^100.
__device__ __forceinline__ i128 floor_uR(float u, i128 R)
{
    const unsigned int b = __float_as_uint(u);
    const int ex = (int)(b >> 23);
    if (!(u > 0.0f) || R <= 0)
        return 0;
    const unsigned long long M = (ex == 0) ? (b & 0x7fffffu) : ((b & 0x7fffffu) | 0x800000u);
    const int sh = (ex == 0) ? 149 : 150 - ex;  // u = M / 2^sh, sh >= 24
    if (sh >= 127)
        return 0;
    return (i128)(((u128)R * M) >> sh);
}

// The exact draw of one job from its NC chunk records (the whole CTA calls
// it; every thread returns the token).  Returns -1 if no weight is positive.
template <int DT>
__device__ int resolve_finish(const RJob &J, int V, const RzRec *recs, const RkRec *kinks,
                              unsigned int kcnt, RFSmem &S, WsHeader *hdr)
{
    const int tid = threadIdx.x;
    const int NC = (V + RCH - 1) / RCH;
    long long at = 0, ad = 0, zt = 0, zd = 0;
    if (tid < NC) {
        const longlong2 r0 = __ldcg(reinterpret_cast<const longlong2 *>(recs + tid));
        const longlong2 r1 = __ldcg(reinterpret_cast<const longlong2 *>(recs + tid) + 1);
        at = r0.x;
        ad = r0.y;
        zt = r1.x;
        zd = r1.y;
    }
    // the listed groups, one per thread, fetched early
    long long get = 0, ged = 0;
    int gc = 0;
    const bool has_group = tid < (int)min(kcnt, (unsigned int)RKCAP);
    if (has_group) {
        const longlong2 e = __ldcg(reinterpret_cast<const longlong2 *>(kinks + tid));
        get = e.x;
        ged = e.y;
        gc = __ldcg(&kinks[tid].chunk);
    }
    bool residual = J.mode == RJ_RESIDUAL;
    unsigned long long Zt = 0, Zd = 0;  // the masses, scaled below 2^62
    if (residual) {
        // exact masses (128-bit), then one common scale
        i128 ta, tb;
        (void)cta_excl_scan((i128)zt, ta, S);
        (void)cta_excl_scan((i128)zd, tb, S);
        const u128 mx = (u128)(ta > tb ? ta : tb);
        const unsigned long long mh = (unsigned long long)(mx >> 64), ml = (unsigned long long)mx;
        const int bits = mh ? 128 - __clzll((long long)mh) : 64 - __clzll((long long)ml);
        const int sc = bits > 62 ? bits - 62 : 0;
        Zt = (unsigned long long)((u128)ta >> sc);
        Zd = (unsigned long long)((u128)tb >> sc);
        const float ratio = __fdiv_rn(__ull2float_rn(Zd), __ull2float_rn(Zt));
        const float rhat = __fdiv_rn(J.rzt, J.rzd);  // the fp32 masses' Z_d / Z_t
        const bool ratio_ok = fabsf(__fdiv_rn(ratio, rhat) - 1.0f) <= RRATIO_TOL;
        const bool sorted_ok = ratio_ok && kcnt <= (unsigned int)RKCAP;
        if (tid == 0 && !ratio_ok)
            atomicAdd(&hdr->n_slow_ratio, 1u);
        if (tid == 0 && kcnt > (unsigned int)RKCAP)
            atomicAdd(&hdr->n_slow_kinks, 1u);
        if (sorted_ok) {
            if (tid < NC) {
                const i128 d = (i128)((u128)(unsigned long long)at * Zd) -
                               (i128)((u128)(unsigned long long)ad * Zt);
                const i128 wc = d >> RSHIFT;
                S.W[tid][0] = lo64(wc);
                S.W[tid][1] = hi64(wc);
            }
            __syncthreads();
            // the groups of undecided elements, weighed with the exact masses
            // and added to their chunks (integer sums: any order gives the
            // same result; 64-bit atomics with the carry done by hand)
            if (has_group) {
                const i128 d = (i128)((u128)(unsigned long long)get * Zd) -
                               (i128)((u128)(unsigned long long)ged * Zt);
                if (d > 0) {
                    const i128 wg = d >> RSHIFT;
                    const unsigned long long lo = lo64(wg), hi = hi64(wg);
                    const unsigned long long old = atomicAdd(&S.W[gc][0], lo);
                    const unsigned long long carry = (old + lo < old) ? 1ull : 0ull;
                    atomicAdd(&S.W[gc][1], hi + carry);
                }
            }
        } else {
            // the sort was not safe (fp32 ratio too far off, or too many
            // undecided elements): every chunk again with the exact masses
            for (int c = 0; c < NC; ++c) {
                i128 w[RFPT];
                rj_weights4<DT>(J, c * RCH + tid * RFPT, V, true, Zt, Zd, w, S.tab);
                i128 s = 0;
#pragma unroll
                for (int i = 0; i < RFPT; ++i)
                    s += w[i];
                i128 tot;
                (void)cta_excl_scan(s, tot, S);
                if (tid == 0) {
                    S.W[c][0] = lo64(tot);
                    S.W[c][1] = hi64(tot);
                }
            }
        }
    } else if (tid < NC) {
        S.W[tid][0] = (unsigned long long)zt;
        S.W[tid][1] = 0ull;
    }
    __syncthreads();

    for (int attempt = 0; attempt < 2; ++attempt) {
        // prefix over chunks; the crossing chunk is the first positive one
        // whose running mass exceeds floor(u * R)
        const i128 w0 = (tid < NC) ? mk128(S.W[tid][0], S.W[tid][1]) : (i128)0;
        i128 R;
        const i128 ex = cta_excl_scan(w0, R, S);
        if (!(R > 0)) {
            if (residual) {
                // the residual vanished (rounding only): draw from the target row
                residual = false;
                if (tid < NC) {
                    S.W[tid][0] = (unsigned long long)zt;
                    S.W[tid][1] = 0ull;
                }
                __syncthreads();
                continue;
            }
            return -1;
        }
        const i128 theta = floor_uR(J.u, R);
        if (tid == 0) {
            S.cstar = INT_MAX;
            S.tok = INT_MAX;
            S.lastp = -1;
        }
        __syncthreads();
        const bool mine = w0 > 0 && ex + w0 > theta;
        if (mine)
            atomicMin(&S.cstar, tid);
        __syncthreads();
        if (S.cstar == INT_MAX) {
            // floor(u * R) at or past the total: the last positive chunk
            // (cannot happen for u < 1; kept as a guard)
            if (tid == 0) {
                i128 b = 0, bl = 0;
                int last = 0;
                for (int c = 0; c < NC; ++c) {
                    const i128 wc = mk128(S.W[c][0], S.W[c][1]);
                    if (wc > 0) {
                        last = c;
                        bl = b;
                    }
                    b += wc;
                }
                S.cstar = last;
                S.before[0] = lo64(bl);
                S.before[1] = hi64(bl);
            }
        } else if (mine && tid == S.cstar) {
            S.before[0] = lo64(ex);
            S.before[1] = hi64(ex);
        }
        __syncthreads();
        const int cs = S.cstar;
        // the crossing chunk, element by element in index order
        i128 w[RFPT];
        rj_weights4<DT>(J, cs * RCH + tid * RFPT, V, residual, Zt, Zd, w, S.tab);
        i128 s = 0;
#pragma unroll
        for (int i = 0; i < RFPT; ++i)
            s += w[i];
        i128 tot;
        const i128 exv = cta_excl_scan(s, tot, S);
        i128 run = mk128(S.before[0], S.before[1]) + exv;
        int cand = INT_MAX, lastp = -1;
#pragma unroll
        for (int i = 0; i < RFPT; ++i) {
            if (w[i] > 0) {
                run += w[i];
                lastp = cs * RCH + tid * RFPT + i;
                if (cand == INT_MAX && run > theta)
                    cand = lastp;
            }
        }
        if (cand != INT_MAX)
            atomicMin(&S.tok, cand);
        if (lastp >= 0)
            atomicMax(&S.lastp, lastp);
        __syncthreads();
        // a threshold past the chunk's element sum (the chunk mass and the
        // element sum differ by the 2^-40 rounding of each product): its
        // last positive weight
        const int tok = (S.tok != INT_MAX) ? S.tok : S.lastp;
        __syncthreads();
        return tok;
    }
    return -1;
}

// ------------------------------------------------------------ the kernels
//
// Listed rows are drawn again in two kernels: the chunk pass (work items
// (listed row, chunk of 2048 elements), handed out by a counter over a
// persistent grid) and the finishing (one CTA per listed row).  The list,
// its records and the counters live in the caller's workspace; the first
// kernel of each call zeroes hdr->n_flag and hdr->next_resolve.

struct RParams {
    WsHeader *hdr;
    const RJob *rjob;      // [cap] the listed draws (count in hdr->n_flag)
    RkRec *rkink;          // [cap][RKCAP] groups of undecided elements
    unsigned int *rkcnt;   // [cap] their counts (zeroed when listed)
    RzRec *rrec;           // [cap][RNC] chunk records
    int RNC, V;
    int32_t *out;          // the token goes to out[out_pos]
    int32_t *out_draw;     // nullable [B][4]: the exact token goes to out_draw[4b + 2]
};

template <int DT>
__global__ void __launch_bounds__(RTH, 3) resolve_chunks_kernel(const RParams P)
{
    __shared__ RSmem S;
    const int tid = threadIdx.x;
    load_exp2_table(S.tab);
    allow_next_kernel();     // the finishing kernel may launch; it waits for this grid
    wait_previous_kernel();  // the list comes from the previous kernel
    const unsigned int nf = *reinterpret_cast<volatile unsigned int *>(&P.hdr->n_flag);
    const long long NC = P.RNC;
    const long long items = (long long)nf * NC;
    // items are handed out by a counter (the first gridDim.x implicitly)
    long long it = blockIdx.x;
    __syncthreads();
    while (it < items) {
        const int f = (int)(it / NC);
        const int q = (int)(it - (long long)f * NC);
        if (tid == 0)
            S.next = (long long)gridDim.x + (long long)atomicAdd(&P.hdr->next_resolve, 1u);
        if (tid < (int)(sizeof(RJob) / 16))
            reinterpret_cast<uint4 *>(&S.job)[tid] =
                __ldcg(reinterpret_cast<const uint4 *>(P.rjob + f) + tid);
        __syncthreads();
        const long long nx = S.next;  // read here: thread 0 rewrites it next iteration
        resolve_chunk<DT>(S.job, q, P.V, P.rrec + (size_t)f * NC + q,
                          P.rkink + (size_t)f * RKCAP, P.rkcnt + f, S);
        __syncthreads();
        it = nx;
    }
}

template <int DT>
__global__ void __launch_bounds__(RFTH, 1) resolve_final_kernel(const RParams P)
{
    __shared__ RFSmem S;
    __shared__ RJob job;
    const int tid = threadIdx.x;
    load_exp2_table(S.tab);
    wait_previous_kernel();  // chunk records come from the chunk pass
    const unsigned int nf = *reinterpret_cast<volatile unsigned int *>(&P.hdr->n_flag);
    const long long NC = P.RNC;
    for (unsigned int f = blockIdx.x; f < nf; f += gridDim.x) {
        if (tid < (int)(sizeof(RJob) / 16))
            reinterpret_cast<uint4 *>(&job)[tid] =
                __ldcg(reinterpret_cast<const uint4 *>(P.rjob + f) + tid);
        __syncthreads();
        const unsigned int kc = __ldcg(P.rkcnt + f);
        const int tok = resolve_finish<DT>(job, P.V, P.rrec + (size_t)f * NC,
                                           P.rkink + (size_t)f * RKCAP, kc, S, P.hdr);
        if (tid == 0) {
            if (tok >= 0)
                P.out[job.out_pos] = tok;
            if (P.out_draw)
                P.out_draw[(size_t)job.b * 4 + 2] = tok;
        }
        __syncthreads();
    }
}

// Launches both kernels on `st` as programmatic dependents of the kernel
// before them (plainly ordered when `pdl` is false).  grid_chunks CTAs of the
// chunk pass, grid_final of the finishing.
template <int DT>
inline cudaError_t launch_resolve(const RParams &P, unsigned int grid_chunks,
                                  unsigned int grid_final, cudaStream_t st, bool pdl)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_chunks);
    cfg.blockDim = dim3(RTH);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, resolve_chunks_kernel<DT>, P);
    if (e != cudaSuccess)
        return e;
    cfg.gridDim = dim3(grid_final);
    cfg.blockDim = dim3(RFTH);
    return cudaLaunchKernelEx(&cfg, resolve_final_kernel<DT>, P);
}

// Workspace bytes for the exact draws of up to `cap` listed rows of V
// elements: their records, counts, groups (residual draws only) and chunk
// records.
inline size_t resolve_bytes(size_t cap, int V, bool residual)
{
    const size_t rnc = ((size_t)V + RCH - 1) / RCH;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    return up(cap * sizeof(RJob)) + up(cap * 4) +
           (residual ? up(cap * RKCAP * sizeof(RkRec)) : 0) + up(cap * rnc * sizeof(RzRec));
}

// The exact-draw regions of a workspace starting at `base` (from resolve_bytes).
inline void resolve_regions(RParams &P, void *base, size_t cap, int V, bool residual)
{
    const size_t rnc = ((size_t)V + RCH - 1) / RCH;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    uint8_t *w = reinterpret_cast<uint8_t *>(base);
    P.rjob = reinterpret_cast<const RJob *>(w);
    w += up(cap * sizeof(RJob));
    P.rkcnt = reinterpret_cast<unsigned int *>(w);
    w += up(cap * 4);
    P.rkink = residual ? reinterpret_cast<RkRec *>(w) : nullptr;
    w += residual ? up(cap * RKCAP * sizeof(RkRec)) : 0;
    P.rrec = reinterpret_cast<RzRec *>(w);
    P.RNC = (int)rnc;
    P.V = V;
}

}  // namespace spec_dev
