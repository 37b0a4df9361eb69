// device_common.cuh -- device helpers shared by the verification and the
// sampling kernels: mbarrier and bulk-copy wrappers with bounded waits,
// packed f32x2 arithmetic, the fp32/bf16 traits that read 16-byte vectors of
// logits, and reads of a row segment staged in shared memory.
#pragma once

#include <cuda_runtime.h>
#include <float.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "spec_verify.h"

namespace spec_dev {

constexpr float LOG2E = 1.4426950408889634f;
constexpr unsigned long long WAIT_NS = 2000000000ull;  // 2 s bound on any wait

// First 256 bytes of every workspace: the device status word (SPEC_DEV_*).
struct WsHeader {
    int status;
    unsigned int next_item;   // row counter of the window filter kernel (zeroed by the first kernel)
    unsigned int next_item2;  // chunk counter of the radix filter kernel (likewise)
    unsigned int n_flag;      // rows listed for an exact draw (likewise)
    unsigned int next_resolve;  // work-item counter of the exact draws (likewise)
    unsigned int n_slow_ratio;  // exact draws whose fp32 mass ratio was too far off (diagnostic)
    unsigned int n_slow_kinks;  // exact draws with too many undecided elements (diagnostic)
    unsigned int n_stream_rows; // filtered rows the group-maximum cut left to the streaming filter
    unsigned int n_radix_rows;  // filtered rows left to the radix kernel
    unsigned int n_stream_draws;  // filtered draws left to the streaming draw kernel
    unsigned int pad[54];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max that propagates NaN, so a NaN logit poisons the row maximum
__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Packed pairs of fp32 values (Blackwell f32x2 arithmetic).  add/mul .rn round
// each half exactly like the scalar instructions, so packing changes no result.
__device__ __forceinline__ unsigned long long f2(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ unsigned long long f2_bits(uint32_t lo, uint32_t hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

__device__ __forceinline__ void f2_split(unsigned long long v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// 2^((x - m) * c) for both halves; x - m is computed as x + (-m), which IEEE
// defines to be the same operation.
__device__ __forceinline__ void exp_pair(unsigned long long x2, unsigned long long negm2,
                                         unsigned long long c2, float &e0, float &e1)
{
    float a0, a1;
    f2_split(mul2(add2(x2, negm2), c2), a0, a1);
    e0 = ex2(a0);
    e1 = ex2(a1);
}

// NaN-propagating maximum of two pairs of bf16 values (exact)
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Programmatic dependent launch: a kernel launched after another on the same
// stream with programmatic serialisation may start early; it must wait here
// before it reads what the previous kernel wrote.
__device__ __forceinline__ void wait_previous_kernel()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next kernel on the stream begin launching (its CTAs still wait in
// wait_previous_kernel until this grid has finished).
__device__ __forceinline__ void allow_next_kernel()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete: false once
// `limit_ns` of global time has passed without it.
__device__ __forceinline__ bool mbar_wait_for(unsigned long long *bar, uint32_t parity,
                                              unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (globaltimer() - t0 > limit_ns)
            return false;
    }
}

// The kernels' wait: bounded by WAIT_NS.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity)
{
    return mbar_wait_for(bar, parity, WAIT_NS);
}

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              unsigned long long *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_addr(p)));
    return r;
}

// ------------------------------------------------------------ dtype traits

template <int DT>
struct Lg;

template <>
struct Lg<SPEC_F32> {
    static constexpr int ES = 4;
    static constexpr int VEC = 4;
    static constexpr uint32_t NEG_INF_WORD = 0xff800000u;
    __device__ static __forceinline__ void unpack(const uint4 &r, float (&x)[VEC])
    {
        x[0] = __uint_as_float(r.x);
        x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z);
        x[3] = __uint_as_float(r.w);
    }
    __device__ static __forceinline__ uint32_t bits_at(const uint8_t *p)
    {
        return *reinterpret_cast<const uint32_t *>(p);
    }
    __device__ static __forceinline__ float load1(const void *base, size_t idx)
    {
        return __ldg(reinterpret_cast<const float *>(base) + idx);
    }
    // maximum of the vector's elements, NaN if any is NaN
    __device__ static __forceinline__ float vmax(const uint4 &r)
    {
        const float a = fmax_nan(__uint_as_float(r.x), __uint_as_float(r.y));
        return fmax_nan(a, fmax_nan(__uint_as_float(r.z), __uint_as_float(r.w)));
    }
    // e[j] = 2^((x_j - m) * c), element by element as expsum2 computes them
    __device__ static __forceinline__ void exp2_vec(const uint4 &r, float negm,
                                                    unsigned long long c2, float (&e)[VEC])
    {
        const unsigned long long negm2 = f2(negm, negm);
        exp_pair(f2_bits(r.x, r.y), negm2, c2, e[0], e[1]);
        exp_pair(f2_bits(r.z, r.w), negm2, c2, e[2], e[3]);
    }
    // sums of 2^((x-m)*c) over the vector as a pair (e0 + e2, e1 + e3)
    __device__ static __forceinline__ unsigned long long expsum2(const uint4 &r, float negm,
                                                                 unsigned long long c2)
    {
        const unsigned long long negm2 = f2(negm, negm);
        float e0, e1, e2, e3;
        exp_pair(f2_bits(r.x, r.y), negm2, c2, e0, e1);
        exp_pair(f2_bits(r.z, r.w), negm2, c2, e2, e3);
        return add2(f2(e0, e1), f2(e2, e3));
    }
    template <int N>
    __device__ static __forceinline__ float tile_max(const uint4 (&raw)[N])
    {
        float m = vmax(raw[0]);
#pragma unroll
        for (int u = 1; u < N; ++u)
            m = fmax_nan(m, vmax(raw[u]));
        return m;
    }
    // place element j's bit pattern into a raw vector
    __device__ static __forceinline__ void put(uint4 &r, int j, uint32_t bits)
    {
        if (j == 0) r.x = bits;
        else if (j == 1) r.y = bits;
        else if (j == 2) r.z = bits;
        else r.w = bits;
    }
};

template <>
struct Lg<SPEC_BF16> {
    static constexpr int ES = 2;
    static constexpr int VEC = 8;
    static constexpr uint32_t NEG_INF_WORD = 0xff80ff80u;
    __device__ static __forceinline__ void unpack(const uint4 &r, float (&x)[VEC])
    {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ uint32_t bits_at(const uint8_t *p)
    {
        return *reinterpret_cast<const uint16_t *>(p);
    }
    __device__ static __forceinline__ float load1(const void *base, size_t idx)
    {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(base) + idx);
        return __uint_as_float(((uint32_t)h) << 16);
    }
    // maximum of the vector's elements, NaN if any is NaN (bf16 maxima are exact)
    __device__ static __forceinline__ float vmax(const uint4 &r)
    {
        const uint32_t h = bmax2_nan(bmax2_nan(r.x, r.y), bmax2_nan(r.z, r.w));
        return fmax_nan(__uint_as_float(h << 16), __uint_as_float(h & 0xffff0000u));
    }
    // x - m for both halves of a word: each bf16 half is widened exactly and
    // added to -m with one rounding, as the fp32 subtraction would do
    __device__ static __forceinline__ unsigned long long sub_pair(uint32_t w, float negm)
    {
        float lo, hi;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "add.rn.f32.bf16 %0, l, %3;\n\tadd.rn.f32.bf16 %1, h, %3;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(w), "f"(negm));
        return f2(lo, hi);
    }
    __device__ static __forceinline__ unsigned long long exp2_pair(uint32_t w, float negm,
                                                                   unsigned long long c2)
    {
        float a0, a1;
        f2_split(mul2(sub_pair(w, negm), c2), a0, a1);
        return f2(ex2(a0), ex2(a1));
    }
    // e[j] = 2^((x_j - m) * c), element by element as expsum2 computes them
    __device__ static __forceinline__ void exp2_vec(const uint4 &r, float negm,
                                                    unsigned long long c2, float (&e)[VEC])
    {
        const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f2_split(exp2_pair(wd[i], negm, c2), e[2 * i], e[2 * i + 1]);
    }
    // sums of 2^((x-m)*c) over the vector as a pair:
    // ((e0+e4) + (e2+e6), (e1+e5) + (e3+e7))
    __device__ static __forceinline__ unsigned long long expsum2(const uint4 &r, float negm,
                                                                 unsigned long long c2)
    {
        const unsigned long long a = add2(exp2_pair(r.x, negm, c2), exp2_pair(r.z, negm, c2));
        const unsigned long long b = add2(exp2_pair(r.y, negm, c2), exp2_pair(r.w, negm, c2));
        return add2(a, b);
    }
    // NaN-propagating maximum over a whole tile's vectors, kept packed
    template <int N>
    __device__ static __forceinline__ float tile_max(const uint4 (&raw)[N])
    {
        uint32_t h = bmax2_nan(bmax2_nan(raw[0].x, raw[0].y), bmax2_nan(raw[0].z, raw[0].w));
#pragma unroll
        for (int u = 1; u < N; ++u)
            h = bmax2_nan(h, bmax2_nan(bmax2_nan(raw[u].x, raw[u].y), bmax2_nan(raw[u].z, raw[u].w)));
        return fmax_nan(__uint_as_float(h << 16), __uint_as_float(h & 0xffff0000u));
    }
    __device__ static __forceinline__ uint32_t merge(uint32_t word, int j, uint32_t bits)
    {
        const int sh = (j & 1) * 16;
        return (word & ~(0xffffu << sh)) | ((bits & 0xffffu) << sh);
    }
    __device__ static __forceinline__ void put(uint4 &r, int j, uint32_t bits)
    {
        const int w = j >> 1;
        if (w == 0) r.x = merge(r.x, j, bits);
        else if (w == 1) r.y = merge(r.y, j, bits);
        else if (w == 2) r.z = merge(r.z, j, bits);
        else r.w = merge(r.w, j, bits);
    }
};

__device__ __forceinline__ uint4 neg_inf_vec(uint32_t word)
{
    return make_uint4(word, word, word, word);
}

// ------------------------------------------------------- softmax partials
//
// A partial is (m, s, idx): maximum, sum of 2^((x-m)*c) relative to that
// maximum, lowest index attaining it.  Combining rescales the smaller side.

__device__ __forceinline__ float rescale(float s, float m_from, float m_to, float c)
{
    return (m_from == -INFINITY) ? 0.0f : s * ex2((m_from - m_to) * c);
}

// Warp-wide combine of per-lane partials (butterfly; every lane ends with the
// same result).  The order depends only on lane numbers.  Sampling partials
// carry (m, s), greedy partials (m, idx).
__device__ __forceinline__ void warp_combine(float &m, float &s, int &idx, float c, bool with_sum)
{
    float mw = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mw = fmax_nan(mw, __shfl_xor_sync(0xffffffffu, mw, o));
    if (with_sum) {
        float sr = rescale(s, m, mw, c);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            sr += __shfl_xor_sync(0xffffffffu, sr, o);
        s = sr;
        idx = INT_MAX;
    } else {
        int cand = (m == mw) ? idx : INT_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
        idx = cand;
    }
    m = mw;
}


// ------------------------------------------------------------ tile loading
//
// A slot holds the 16-byte-aligned byte range around one row segment.  Vector
// v (row-relative, VEC elements) is read with one 16-byte shared load when the
// segment starts on a 16-byte boundary and was copied whole; otherwise element
// by element, from the slot or, past the copied bytes (only at the very end of
// an array), from global memory.  Elements outside [e0, e1) read as -inf.

struct Seg {
    const uint8_t *slot;
    const void *arr;
    size_t row;
    int V;
    int e0, e1, phase, ncopied;
    bool fast;
};

template <int DT>
__device__ __forceinline__ Seg make_seg(const uint8_t *slot, const void *arr, size_t row, int V,
                                        int e0, int e1, int phase, int ncopied)
{
    using L = Lg<DT>;
    Seg g;
    g.slot = slot;
    g.arr = arr;
    g.row = row;
    g.V = V;
    g.e0 = e0;
    g.e1 = e1;
    g.phase = phase;
    g.ncopied = ncopied;
    const int nbytes = (e1 - e0) * L::ES;
    g.fast = (phase == 0) && ((nbytes & 15) == 0) && (ncopied >= nbytes);
    return g;
}

template <int DT>
__device__ __forceinline__ uint4 seg_vec(const Seg &g, int v)
{
    using L = Lg<DT>;
    if (g.fast && v * L::VEC >= g.e0 && (v + 1) * L::VEC <= g.e1)
        return ld_shared_v4(g.slot + (size_t)(v * L::VEC - g.e0) * L::ES);
    uint4 r = neg_inf_vec(L::NEG_INF_WORD);
#pragma unroll
    for (int j = 0; j < L::VEC; ++j) {
        const int e = v * L::VEC + j;
        if (e >= g.e0 && e < g.e1) {
            const int off = g.phase + (e - g.e0) * L::ES;
            uint32_t bits;
            if (off + L::ES <= g.ncopied)
                bits = L::bits_at(g.slot + off);
            else
                bits = __float_as_uint(L::load1(g.arr, g.row * (size_t)g.V + e)) >> (DT == SPEC_BF16 ? 16 : 0);
            L::put(r, j, bits);
        }
    }
    return r;
}

// Row vector straight from global memory (through L2), for chunk searches.
template <int DT>
__device__ __forceinline__ uint4 row_vec(const void *arr, size_t row, int v, int V)
{
    using L = Lg<DT>;
    const int e = v * L::VEC;
    const uint8_t *base = reinterpret_cast<const uint8_t *>(arr) + row * (size_t)V * L::ES;
    if (e + L::VEC <= V && (reinterpret_cast<uintptr_t>(base) & 15) == 0)
        return __ldcg(reinterpret_cast<const uint4 *>(base) + v);
    uint4 r = neg_inf_vec(L::NEG_INF_WORD);
#pragma unroll
    for (int j = 0; j < L::VEC; ++j)
        if (e + j < V)
            L::put(r, j, __float_as_uint(L::load1(base, (size_t)(e + j))) >> (DT == SPEC_BF16 ? 16 : 0));
    return r;
}


__device__ __forceinline__ bool temperature_valid(float T)
{
    return !(isnan(T) || T < 0.0f || isinf(T) || (T > 0.0f && T < FLT_MIN));
}

// ------------------------------------------------------ draws from chunk records
//
// A row summarised by chunk records: chunk q is the contiguous 4 KB of the row
// starting at byte 4096*q (lane l of the chunk holds its 16-byte vectors
// 256*q + 32*u + l, u < CHUNK_UV), and its record is (M_q, S_q) = the chunk
// maximum and the sum of 2^((x - M_q) * c) over it.

constexpr int CHUNK_BYTES = 4096;
constexpr int CHUNK_UV = CHUNK_BYTES / (32 * 16);  // vectors per lane per chunk

// Inclusive Kogge-Stone scan of one value per lane.
__device__ __forceinline__ float lane_scan(float x, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x = x + y;
    }
    return x;
}

// Inverse-CDF draw with uniform u from weights 2^((x - m) * c), m the row
// maximum, for one row given its NC chunk records (one warp; every lane gets
// the result).  C(x) runs over the chunks' scaled sums S_q * 2^((M_q - m) * c)
// in chunk order, then, inside the crossing chunk (read again from `logits`),
// over its elements in index order; the token is the smallest x with
// C(x) > u * R.  A threshold that rounding leaves past a running total takes
// the last positive weight before it.  Returns -1 if no weight is positive.
// *near (every lane) is set when u * R lies within guard * R of the chosen
// cell's edges as computed here, or a rounding fallback was taken: the fp32
// sums cannot tell such a draw apart from its neighbour's.
template <int DT>
__device__ int records_draw(const float2 *rc, int NC, float m, float c, float u,
                            const void *logits, size_t row, int V, int lane, float guard,
                            bool &near, float *gap_u = nullptr)
{
    near = false;
    if (gap_u)
        *gap_u = 0.0f;
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    constexpr int RC = 8;  // records a lane keeps in registers
    const int per = (NC + 31) / 32;
    const int c0 = min(NC, lane * per), c1 = min(NC, c0 + per);
    const bool cached = per <= RC;
    float2 cache[RC];
#pragma unroll
    for (int i = 0; i < RC; ++i)
        cache[i] = (cached && c0 + i < c1) ? __ldcg(rc + c0 + i) : make_float2(-INFINITY, 0.0f);
    auto rec_at = [&](int i) -> float2 {  // the lane's i-th record
        if (cached) {
            float2 f = cache[0];
#pragma unroll
            for (int t = 1; t < RC; ++t)
                if (t == i)
                    f = cache[t];
            return f;
        }
        return __ldcg(rc + c0 + i);
    };

    // running totals of the scaled chunk sums (each lane a contiguous range,
    // then a scan over lanes); R = the last
    float sl = 0.0f;
    if (cached) {
#pragma unroll
        for (int i = 0; i < RC; ++i)
            if (c0 + i < c1)
                sl += rescale(cache[i].y, cache[i].x, m, c);
    } else {
        for (int q = c0; q < c1; ++q) {
            const float2 f = __ldcg(rc + q);
            sl += rescale(f.y, f.x, m, c);
        }
    }
    const float incl = lane_scan(sl, lane);
    const float Rtot = __shfl_sync(0xffffffffu, incl, 31);
    const float theta = u * Rtot;
    const unsigned cross = __ballot_sync(0xffffffffu, incl > theta);
    int Lw;
    if (cross) {
        Lw = __ffs(cross) - 1;
    } else {
        const unsigned pos = __ballot_sync(0xffffffffu, sl > 0.0f);
        Lw = pos ? 31 - __clz(pos) : -1;
    }
    if (Lw < 0)
        return -1;

    // the crossing lane walks its chunks from the running total before it
    const float before_lane = __shfl_sync(0xffffffffu, incl, Lw > 0 ? Lw - 1 : 0);
    int chunk = -1;
    float cbefore = 0.0f, Mc = 0.0f;
    if (lane == Lw) {
        float C = (Lw > 0) ? before_lane : 0.0f;
        int lastpos = -1;
        float lastC = 0.0f, lastM = 0.0f;
        for (int i = 0; i < c1 - c0 && chunk < 0; ++i) {
            const float2 f = rec_at(i);
            const float w = rescale(f.y, f.x, m, c);
            if (w > 0.0f) {
                if (C + w > theta) {
                    chunk = c0 + i;
                    cbefore = C;
                    Mc = f.x;
                } else {
                    lastpos = c0 + i;
                    lastC = C;
                    lastM = f.x;
                }
            }
            C += w;
        }
        if (chunk < 0) {  // rounding left the threshold past the lane's total
            chunk = lastpos;
            cbefore = lastC;
            Mc = lastM;
            near = true;
        }
    }
    near = __shfl_sync(0xffffffffu, near ? 1 : 0, Lw) != 0 || !cross;
    chunk = __shfl_sync(0xffffffffu, chunk, Lw);
    if (chunk < 0)
        return -1;
    cbefore = __shfl_sync(0xffffffffu, cbefore, Lw);
    Mc = __shfl_sync(0xffffffffu, Mc, Lw);

    // the chunk again (all its vectors in one round trip), in index order, in
    // units of 2^((x - Mc) * c)
    const int vb = chunk * (32 * CHUNK_UV);
    uint4 raw[CHUNK_UV];
#pragma unroll
    for (int uv = 0; uv < CHUNK_UV; ++uv)
        raw[uv] = row_vec<DT>(logits, row, vb + uv * 32 + lane, V);
    const float csc = ex2((Mc - m) * c);
    const float tloc = (theta - cbefore) / csc;
    const float gloc = guard * (Rtot / csc);  // the guard in the chunk's units
    const unsigned long long c2 = f2(c, c);
    float carry = 0.0f;
    int tok = -1, last_u = -1, last_lane = -1;
#pragma unroll
    for (int uv = 0; uv < CHUNK_UV; ++uv) {
        if (tok >= 0)
            continue;
        const int v = vb + uv * 32 + lane;
        float e[VEC];
        L::exp2_vec(raw[uv], -Mc, c2, e);
        float tau = 0.0f;
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            tau = tau + e[j];
        const float in_l = lane_scan(tau, lane);
        const unsigned hit = __ballot_sync(0xffffffffu, carry + in_l > tloc && tau > 0.0f);
        if (hit) {
            const int hl = __ffs(hit) - 1;
            int t = -1;
            int nr = 0;
            float gl = 0.0f;
            if (lane == hl) {
                float run = carry + (in_l - tau);
                int lastj = -1;
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    if (t < 0 && e[j] > 0.0f) {
                        const float prev = run;
                        run = run + e[j];
                        lastj = j;
                        if (run > tloc) {
                            t = v * VEC + j;
                            nr = (tloc - prev < gloc || run - tloc < gloc) ? 1 : 0;
                            gl = fminf(tloc - prev, run - tloc) * (csc / Rtot);
                        }
                    }
                }
                if (t < 0) {
                    t = v * VEC + lastj;  // rounding within the lane: its last positive weight
                    nr = 1;
                }
            }
            tok = __shfl_sync(0xffffffffu, t, hl);
            near = near || __shfl_sync(0xffffffffu, nr, hl) != 0;
            gl = __shfl_sync(0xffffffffu, gl, hl);
            if (gap_u)
                *gap_u = gl;
        } else {
            const unsigned pos = __ballot_sync(0xffffffffu, tau > 0.0f);
            if (pos) {
                last_u = uv;
                last_lane = 31 - __clz(pos);
            }
            carry = carry + __shfl_sync(0xffffffffu, in_l, 31);
        }
    }
    if (tok < 0 && last_u >= 0) {
        // rounding left the threshold past the chunk's running total: its
        // last positive weight
        int t = -1;
        if (lane == last_lane) {
#pragma unroll
            for (int uv = 0; uv < CHUNK_UV; ++uv) {
                if (uv == last_u) {
                    float e[VEC];
                    L::exp2_vec(raw[uv], -Mc, c2, e);
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        if (e[j] > 0.0f)
                            t = (vb + uv * 32 + lane) * VEC + j;
                }
            }
        }
        tok = __shfl_sync(0xffffffffu, t, last_lane);
        near = true;
    }
    return tok;
}

}  // namespace spec_dev
