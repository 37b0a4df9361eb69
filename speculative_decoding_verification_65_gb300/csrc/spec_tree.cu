// spec_tree.cu -- GB300 (sm_103a) kernel and C ABI for tree verification
// (include/spec_tree.h states the rule and its sources).
//
// One CTA of 16 warps per sequence walks the tree from the root.  At each
// visited node the CTA streams that node's rows once for the softmax
// statistics (row maximum and the sum of 2^((x - m) c), c = log2(e) / T; for
// a greedy sequence the maximum and its lowest index), gathers the children's
// target and draft logits, and runs the sibling tests.  A rejection costs one
// more pass over the node's two rows for the residual mass
// M = sum max(0, p - C q); the pass after the last rejection also serves the
// draw.  Only visited rows are read, so the bytes a sequence moves are its
// path's rows, not the whole tree's.
//
// A pass splits the row into 16 contiguous segments of 16-byte vectors, one
// per warp (lane l takes vectors l, l+32, ... of its warp's segment), so the
// per-warp totals of a residual pass are the row's running mass at segment
// granularity.  For a draw from p_c itself (a leaf's bonus token) the
// statistics pass's per-warp partials already are those totals, and no
// residual pass runs.  The draw takes u * R against the segment totals in
// order, splits the crossing segment into 16 sub-ranges that the 16 warps
// sum at once, and one warp reads the crossing sub-range in index order (a
// Kogge-Stone scan over the 32 lanes of each step, elements left to right
// inside a lane).  A threshold that rounding leaves past a range's own
// running total takes the range's last positive weight, the clamp the
// method's draw already has for the whole row.
//
// The statistics and residual passes stream each warp segment with every
// thread keeping three vectors of each row in flight by cp.async into shared
// memory slots only it reads (no barrier; the copies are waited for with
// cp.async.wait_group, no spin).  CTA x walks the x-th sampled sequence, then
// the greedy ones, so the longer walks start first.
//
// Rows start anywhere: vector a of a row covers the 16-byte-aligned elements
// [A0 + a VEC, A0 + (a+1) VEC) of the array, A0 the row's first element
// rounded down to a multiple of VEC; the elements outside the row read as
// -inf (weight 0), loaded one by one only in the row's first and last vector.
#include <cuda_runtime.h>
#include <float.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "spec_tree.h"
#include "spec_verify.h"
#include "device_common.cuh"

namespace {

using namespace spec_dev;

constexpr int TW = 16;         // warps per CTA
constexpr int TTH = TW * 32;   // threads per CTA (one CTA per sequence, 2 per SM)
constexpr int MAXN = SPEC_TREE_MAX_NODES;

struct TParams {
    const void *target, *draft;
    const int32_t *parent, *tokens, *n_nodes;
    const float *u_accept, *u_resample, *temperature;
    int32_t *out_tokens, *out_nodes, *out_n;
    int N, V;
};

struct TSmem {
    int par[MAXN];
    int tok[MAXN];
    int kids[MAXN];   // children of the current node, in index order
    float r0[MAXN];   // p(x)/q(x) of each child; -1 when q(x) = 0
    int path[MAXN];
    float red_m[TW], red_s[TW], red_s2[TW], red_m2[TW];
    int red_i[TW];
    float wtot[TW];   // per-segment mass of the current draw weights
    float wsub[TW];   // per-warp sub-range masses inside the crossing segment
    int nk, next, pick;
};

// Vector a of the row starting at element `off` (A0 = off rounded down).
template <int DT>
__device__ __forceinline__ uint4 tvec(const void *arr, size_t off, int V, size_t A0, int a)
{
    using L = Lg<DT>;
    const size_t e0 = A0 + (size_t)a * L::VEC;
    if (e0 >= off && e0 + L::VEC <= off + (size_t)V)
        return __ldcg(reinterpret_cast<const uint4 *>(arr) + e0 / L::VEC);
    uint4 r = neg_inf_vec(L::NEG_INF_WORD);
#pragma unroll
    for (int j = 0; j < L::VEC; ++j) {
        const size_t e = e0 + j;
        if (e >= off && e < off + (size_t)V)
            L::put(r, j, __float_as_uint(L::load1(arr, e)) >> (DT == SPEC_BF16 ? 16 : 0));
    }
    return r;
}

constexpr int STG = 3;  // vectors of each row in flight per thread (cp.async stages;
                        // 4 and 6 measured slower: their shared memory costs occupancy)
constexpr size_t RING_BYTES = (size_t)STG * 2 * TTH * 16;  // dynamic shared memory

__device__ __forceinline__ void cp16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

struct Span {
    size_t off, A0;
    int s0, s1;  // this warp's vectors [s0, s1)
};

template <int DT>
__device__ __forceinline__ Span span_of(size_t off, int V, int seg)
{
    using L = Lg<DT>;
    Span s;
    s.off = off;
    s.A0 = off - off % L::VEC;
    const int nvv = (int)((off - s.A0 + (size_t)V + L::VEC - 1) / L::VEC);
    const int per = (nvv + TW - 1) / TW;
    s.s0 = min(nvv, seg * per);
    s.s1 = min(nvv, s.s0 + per);
    return s;
}

// Vectors a, a + 32, ... of a warp segment of one or two rows, each thread
// keeping STG of them in flight with cp.async into slots only it reads (no
// barrier needed; a warp's lanes use consecutive 16 bytes of a slot row, so
// the reads are free of bank conflicts).  Vectors not wholly inside the row
// are read element by element when used.
template <int DT, bool TWO>
struct Stream {
    const void *arr0, *arr1;
    size_t off, A0;
    int V, s1;
    uint8_t *ring;
    int tid;
    __device__ __forceinline__ bool full(int a) const
    {
        using L = Lg<DT>;
        const size_t e0 = A0 + (size_t)a * L::VEC;
        return e0 >= off && e0 + L::VEC <= off + (size_t)V;
    }
    __device__ __forceinline__ uint8_t *slot(int q, int r) const
    {
        return ring + ((size_t)(q * 2 + r) * TTH + tid) * 16;
    }
    __device__ __forceinline__ void issue(int a, int q) const
    {
        using L = Lg<DT>;
        if (a < s1 && full(a)) {
            const size_t vi = (A0 + (size_t)a * L::VEC) / L::VEC;
            cp16(slot(q, 0), reinterpret_cast<const uint4 *>(arr0) + vi);
            if (TWO)
                cp16(slot(q, 1), reinterpret_cast<const uint4 *>(arr1) + vi);
        }
        cp_commit();
    }
    __device__ __forceinline__ void get(int a, int q, uint4 &x0, uint4 &x1) const
    {
        if (full(a)) {
            x0 = ld_shared_v4(slot(q, 0));
            if (TWO)
                x1 = ld_shared_v4(slot(q, 1));
        } else {
            x0 = tvec<DT>(arr0, off, V, A0, a);
            if (TWO)
                x1 = tvec<DT>(arr1, off, V, A0, a);
        }
    }
};

// Streams a warp segment through Stream, calling fn(a, x0, x1) per vector.
template <int DT, bool TWO, typename F>
__device__ __forceinline__ void stream_segment(const Stream<DT, TWO> &st, int s0, int lane, F fn)
{
    const int a0 = s0 + lane;
#pragma unroll
    for (int q = 0; q < STG - 1; ++q)
        st.issue(a0 + 32 * q, q);
    int q = 0;
    for (int a = a0; a < st.s1; a += 32) {
        st.issue(a + 32 * (STG - 1), (q + STG - 1) % STG);
        cp_wait<STG - 1>();
        uint4 x0, x1 = x0;
        st.get(a, q, x0, x1);
        fn(a, x0, x1);
        q = (q + 1 == STG) ? 0 : q + 1;
    }
    cp_wait<0>();
}

template <int DT>
__device__ __forceinline__ void online1(const uint4 &x0, float c, unsigned long long c2, float &m,
                                        float &s, bool &bad)
{
    using L = Lg<DT>;
    const float vm = L::vmax(x0);
    bad |= !(vm < INFINITY);
    if (vm > m) {
        s = rescale(s, m, vm, c);
        m = vm;
    }
    if (m > -INFINITY) {
        float lo, hi;
        f2_split(L::expsum2(x0, -m, c2), lo, hi);
        s += lo + hi;
    }
}

// One online softmax partial (m, s) over a vector pair.
template <int DT>
__device__ __forceinline__ void online2(const uint4 &x0, const uint4 &x1, float c,
                                        unsigned long long c2, float &m, float &s, bool &bad)
{
    using L = Lg<DT>;
    const float vm = fmax_nan(L::vmax(x0), L::vmax(x1));
    bad |= !(vm < INFINITY);
    if (vm > m) {
        s = rescale(s, m, vm, c);
        m = vm;
    }
    if (m > -INFINITY) {
        float lo, hi;
        f2_split(add2(L::expsum2(x0, -m, c2), L::expsum2(x1, -m, c2)), lo, hi);
        s += lo + hi;
    }
}

// Block-wide combine of per-lane (m, s) partials; every thread gets the row's.
__device__ __forceinline__ void block_ms(float &m, float &s, float c, float *rm, float *rs,
                                         int warp, int lane)
{
    int idx = 0;
    warp_combine(m, s, idx, c, true);
    if (lane == 0) {
        rm[warp] = m;
        rs[warp] = s;
    }
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < TW; ++w)
        M = fmax_nan(M, rm[w]);
    float Z = 0.0f;
    for (int w = 0; w < TW; ++w)
        Z += rescale(rs[w], rm[w], M, c);
    m = M;
    s = Z;
}

// Softmax statistics of the target row (and the draft row when TWO).
// Returns true (every thread) if a row read holds NaN or +inf or is all -inf.
template <int DT, bool TWO>
__device__ bool row_stats(const TParams &P, size_t off, float c, TSmem &S, int warp, int lane,
                          float &mt, float &zt, float &md, float &zd, uint8_t *ring)
{
    const Span sp = span_of<DT>(off, P.V, warp);
    const unsigned long long c2 = f2(c, c);
    float m0 = -INFINITY, s0 = 0.0f, m1 = -INFINITY, s1 = 0.0f;
    bool bad = false;
    const Stream<DT, TWO> st{P.target, P.draft, off, sp.A0, P.V, sp.s1, ring, (int)threadIdx.x};
    stream_segment<DT, TWO>(st, sp.s0, lane, [&](int, const uint4 &t0, const uint4 &d0) {
        online1<DT>(t0, c, c2, m0, s0, bad);
        if (TWO)
            online1<DT>(d0, c, c2, m1, s1, bad);
    });
    bad = __syncthreads_or(bad) != 0;
    block_ms(m0, s0, c, S.red_m, S.red_s, warp, lane);
    if (TWO)
        block_ms(m1, s1, c, S.red_m2, S.red_s2, warp, lane);
    mt = m0;
    zt = s0;
    md = m1;
    zd = s1;
    __syncthreads();  // the reduction slots are reused by the next pass
    return bad || m0 == -INFINITY || (TWO && m1 == -INFINITY);
}

// Maximum and lowest index attaining it of the target row (greedy).
template <int DT>
__device__ bool row_argmax(const TParams &P, size_t off, TSmem &S, int warp, int lane,
                           int &arg)
{
    using L = Lg<DT>;
    const Span sp = span_of<DT>(off, P.V, warp);
    float m = -INFINITY;
    int idx = INT_MAX;
    bool bad = false;
    for (int a = sp.s0 + lane; a < sp.s1; a += 32) {
        const uint4 r = tvec<DT>(P.target, off, P.V, sp.A0, a);
        const float vm = L::vmax(r);
        bad |= !(vm < INFINITY);
        if (vm > m) {
            float x[L::VEC];
            L::unpack(r, x);
            int j = L::VEC - 1;
#pragma unroll
            for (int i = L::VEC - 1; i >= 0; --i)
                if (x[i] == vm)
                    j = i;
            m = vm;
            idx = (int)((long long)(sp.A0 + (size_t)a * L::VEC + j) - (long long)off);
        }
    }
    bad = __syncthreads_or(bad) != 0;
    float s = 0.0f;
    warp_combine(m, s, idx, 0.0f, false);
    if (lane == 0) {
        S.red_m[warp] = m;
        S.red_i[warp] = idx;
    }
    __syncthreads();
    float M = -INFINITY;
    int I = INT_MAX;
    for (int w = 0; w < TW; ++w)
        if (S.red_m[w] > M) {  // segments in index order: the first maximum wins
            M = S.red_m[w];
            I = S.red_i[w];
        }
    arg = I;
    __syncthreads();
    return bad || M == -INFINITY;
}

// Weights of one vector: w = max(0, p - C q) with p = 2^((t - mt) c) it,
// q = 2^((d - md) c) id, or w = p when C == 0.  Explicit roundings, so the
// residual pass and the search compute identical weights.
struct Wt {
    float negmt, negmd, it, id, C;
    unsigned long long c2;
};

template <int DT>
__device__ __forceinline__ void weights(const uint4 &t, const uint4 &d, const Wt &w,
                                        float (&out)[Lg<DT>::VEC])
{
    using L = Lg<DT>;
    float et[L::VEC];
    L::exp2_vec(t, w.negmt, w.c2, et);
    if (w.C > 0.0f) {
        float ed[L::VEC];
        L::exp2_vec(d, w.negmd, w.c2, ed);
#pragma unroll
        for (int j = 0; j < L::VEC; ++j)
            out[j] = fmaxf(0.0f, __fmaf_rn(-w.C, __fmul_rn(ed[j], w.id), __fmul_rn(et[j], w.it)));
    } else {
#pragma unroll
        for (int j = 0; j < L::VEC; ++j)
            out[j] = __fmul_rn(et[j], w.it);
    }
}

// Residual pass: S.wtot[w] = the mass of warp w's segment; returns the total
// (sum of the segment totals in segment order), the same in every thread.
template <int DT>
__device__ float residual_pass(const TParams &P, size_t off, const Wt &w, TSmem &S, int warp,
                               int lane, uint8_t *ring)
{
    using L = Lg<DT>;
    const Span sp = span_of<DT>(off, P.V, warp);
    float acc = 0.0f;
    auto add = [&](int, const uint4 &t0, const uint4 &d0) {
        float x0[L::VEC];
        weights<DT>(t0, d0, w, x0);
        float v = 0.0f;
#pragma unroll
        for (int j = 0; j < L::VEC; ++j)
            v += x0[j];
        acc += v;
    };
    if (w.C > 0.0f) {  // residual weights read both rows
        const Stream<DT, true> st{P.target, P.draft, off, sp.A0, P.V, sp.s1, ring, (int)threadIdx.x};
        stream_segment<DT, true>(st, sp.s0, lane, add);
    } else {
        const Stream<DT, false> st{P.target, P.draft, off, sp.A0, P.V, sp.s1, ring, (int)threadIdx.x};
        stream_segment<DT, false>(st, sp.s0, lane, add);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0)
        S.wtot[warp] = acc;
    __syncthreads();
    float R = 0.0f;
    for (int i = 0; i < TW; ++i)
        R += S.wtot[i];
    __syncthreads();  // every thread has read the totals before a next pass rewrites them
    return R;
}

// The range a mass threshold tau falls in, given the ranges' totals in
// order: the first whose running total exceeds tau, else (rounding left tau
// past the end) the last with a positive total; rem = tau minus the mass of
// the ranges before it.  Every thread computes the same.
__device__ __forceinline__ int pick_range(const float *tot, float tau, float &rem)
{
    int sel = -1, last = 0;
    float pre = 0.0f, pre_sel = 0.0f;
    for (int i = 0; i < TW; ++i) {
        if (tot[i] > 0.0f)
            last = i;
        if (sel < 0 && pre + tot[i] > tau) {
            sel = i;
            pre_sel = pre;
        }
        pre += tot[i];
    }
    if (sel < 0) {
        sel = last;
        pre_sel = 0.0f;
        for (int i = 0; i < last; ++i)
            pre_sel += tot[i];
    }
    rem = tau - pre_sel;
    return sel;
}

// The draw with uniform u from the current weights, whose per-segment masses
// are in S.wtot (total R): the segment whose running mass crosses u * R; the
// warp sub-range of that segment that crosses (all warps sum one sub-range
// each); then that sub-range in index order (one warp, a Kogge-Stone scan over
// the lanes of each step, elements left to right in a lane, the next step's
// vectors loaded ahead).  Returns the row element (every thread).
template <int DT>
__device__ int draw_from(const TParams &P, size_t off, const Wt &w, float R, float u, TSmem &S,
                         int warp, int lane)
{
    using L = Lg<DT>;
    const uint4 ninf = neg_inf_vec(L::NEG_INF_WORD);
    const bool with_d = w.C > 0.0f;
    float tau1;
    const int seg = pick_range(S.wtot, u * R, tau1);
    const Span sp = span_of<DT>(off, P.V, seg);
    const int nv = sp.s1 - sp.s0;
    const int sub = (nv + TW - 1) / TW;

    // level 2: warp w sums sub-range w of the segment
    {
        const int a0 = sp.s0 + min(nv, warp * sub), a1 = sp.s0 + min(nv, warp * sub + sub);
        float acc = 0.0f;
        for (int a = a0 + lane; a < a1; a += 32) {
            const uint4 t = tvec<DT>(P.target, off, P.V, sp.A0, a);
            const uint4 d = with_d ? tvec<DT>(P.draft, off, P.V, sp.A0, a) : ninf;
            float x[L::VEC];
            weights<DT>(t, d, w, x);
#pragma unroll
            for (int j = 0; j < L::VEC; ++j)
                acc += x[j];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0)
            S.wsub[warp] = acc;
    }
    __syncthreads();
    float tw;
    const int ss = pick_range(S.wsub, tau1, tw);

    // level 3: warp ss walks its sub-range in index order
    if (warp == ss) {
        const int b0 = sp.s0 + min(nv, ss * sub), b1 = sp.s0 + min(nv, ss * sub + sub);
        float base = 0.0f;
        int found = -1, lastpos = -1;
        uint4 tn = (b0 + lane < b1) ? tvec<DT>(P.target, off, P.V, sp.A0, b0 + lane) : ninf;
        uint4 dn = (with_d && b0 + lane < b1) ? tvec<DT>(P.draft, off, P.V, sp.A0, b0 + lane)
                                                : ninf;
        for (int a0 = b0; a0 < b1; a0 += 32) {
            const int a = a0 + lane;
            const uint4 t = tn, d = dn;
            const int an = a + 32;
            tn = (an < b1) ? tvec<DT>(P.target, off, P.V, sp.A0, an) : ninf;
            dn = (with_d && an < b1) ? tvec<DT>(P.draft, off, P.V, sp.A0, an) : ninf;
            float x[L::VEC];
            weights<DT>(t, d, w, x);
            const int e0 = (int)((long long)(sp.A0 + (size_t)a * L::VEC) - (long long)off);
            float ls = 0.0f;
            int lp = -1;
#pragma unroll
            for (int j = 0; j < L::VEC; ++j) {
                ls += x[j];
                if (x[j] > 0.0f)
                    lp = e0 + j;
            }
            if (lp > lastpos)
                lastpos = lp;
            const float incl = lane_scan(ls, lane);
            float excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0)
                excl = 0.0f;
            const unsigned hit = __ballot_sync(0xffffffffu, base + incl > tw);
            if (hit) {
                const int hl = __ffs(hit) - 1;
                int f = -1;
                if (lane == hl) {
                    float run = base + excl;
#pragma unroll
                    for (int j = 0; j < L::VEC; ++j) {
                        run += x[j];
                        if (f < 0 && run > tw && x[j] > 0.0f)
                            f = e0 + j;
                    }
                    if (f < 0)
                        f = lp;
                }
                found = __shfl_sync(0xffffffffu, f, hl);
                break;
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (found < 0) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
            found = lastpos;
        }
        if (lane == 0)
            S.pick = found;
    }
    __syncthreads();
    const int x = S.pick;
    __syncthreads();
    return x;
}

// The sequence CTA x walks: the sampled sequences (T != 0) first, in index
// order, then the greedy ones.  CTAs start roughly in index order, and a
// sampled walk reads two rows per node and a residual per rejection where a
// greedy walk reads one row, so the longer walks start first and the shorter
// ones fill the tail (longest first).  Every CTA reads the batch's
// temperatures, so the order costs O(B^2) loads in all: batches above
// ORDER_MAX keep the index order.
constexpr int ORDER_MAX = 2048;

__device__ int walk_order(const TParams &P, TSmem &S, int tid, int warp, int lane)
{
    const int x = blockIdx.x, nb = (int)gridDim.x;
    if (nb > ORDER_MAX)
        return x;
    // block-wide count of the sequences matching `sampled` in [c0, c0 + TTH)
    auto count = [&](int c0, bool sampled, int &excl) -> int {
        const int i = c0 + tid;
        const bool m = i < nb && ((P.temperature[i] != 0.0f) == sampled);
        const unsigned int bm = __ballot_sync(0xffffffffu, m);
        if (lane == 0)
            S.red_i[warp] = __popc(bm);
        __syncthreads();
        int before = 0, tot = 0;
        for (int w = 0; w < TW; ++w) {
            before += (w < warp) ? S.red_i[w] : 0;
            tot += S.red_i[w];
        }
        __syncthreads();
        excl = before + __popc(bm & ((1u << lane) - 1u));
        return tot;
    };
    int ns = 0, ex;
    for (int c0 = 0; c0 < nb; c0 += TTH)
        ns += count(c0, true, ex);
    const bool sampled = x < ns;
    const int rank = sampled ? x : x - ns;
    int base = 0;
    for (int c0 = 0; c0 < nb; c0 += TTH) {
        const int tot = count(c0, sampled, ex);
        const int i = c0 + tid;
        if (i < nb && ((P.temperature[i] != 0.0f) == sampled) && base + ex == rank)
            S.pick = i;
        base += tot;
        if (base > rank)
            break;  // the same in every thread
    }
    __syncthreads();
    const int b = S.pick;
    __syncthreads();
    return b;
}

template <int DT>
__global__ void __launch_bounds__(TTH, 2) tree_kernel(const TParams P)
{
    __shared__ TSmem S;
    extern __shared__ __align__(16) uint8_t ring[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = walk_order(P, S, tid, warp, lane);
    const int N = P.N, V = P.V;
    const float T = P.temperature[b];
    const bool greedy = (T == 0.0f);
    const int n = P.n_nodes[b];
    bool bad = !temperature_valid(T) || n < 1 || n > N;
    if (!bad) {
        for (int i = tid; i < n; i += TTH) {
            const int p = (i == 0) ? -1 : P.parent[(size_t)b * N + i];
            const int t = (i == 0) ? -1 : P.tokens[(size_t)b * N + i];
            if (i > 0 && (p < 0 || p >= i || t < 0 || t >= V))
                bad = true;
            S.par[i] = p;
            S.tok[i] = t;
        }
    }
    bool err = __syncthreads_or(bad) != 0;
    const float c = (!err && !greedy) ? LOG2E / T : 0.0f;

    int cur = 0, depth = 0, token = -1;
    while (!err) {
        // children of the current node, in index order (warp 0, ballot compaction)
        if (warp == 0) {
            int cnt = 0;
            for (int base = cur + 1; base < n; base += 32) {
                const int i = base + lane;
                const bool is = i < n && S.par[i] == cur;
                const unsigned m = __ballot_sync(0xffffffffu, is);
                if (is)
                    S.kids[cnt + __popc(m & ((1u << lane) - 1u))] = i;
                cnt += __popc(m);
            }
            if (lane == 0)
                S.nk = cnt;
        }
        __syncthreads();
        const int nk = S.nk;
        const size_t off = ((size_t)b * N + cur) * (size_t)V;
        int next = -1;
        if (greedy) {
            int arg = 0;
            if (row_argmax<DT>(P, off, S, warp, lane, arg)) {
                err = true;
                break;
            }
            if (warp == 0) {
                int f = INT_MAX;
                for (int i = lane; i < nk; i += 32)
                    if (S.tok[S.kids[i]] == arg)
                        f = min(f, i);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    f = min(f, __shfl_xor_sync(0xffffffffu, f, o));
                if (lane == 0)
                    S.next = (f == INT_MAX) ? -1 : S.kids[f];
            }
            __syncthreads();
            next = S.next;
            if (next < 0) {
                token = arg;
                break;
            }
        } else {
            float mt, zt, md = 0.0f, zd = 1.0f;
            const bool rowbad =
                (nk > 0) ? row_stats<DT, true>(P, off, c, S, warp, lane, mt, zt, md, zd, ring)
                         : row_stats<DT, false>(P, off, c, S, warp, lane, mt, zt, md, zd, ring);
            if (rowbad) {
                err = true;
                break;
            }
            Wt w;
            w.negmt = -mt;
            w.negmd = -md;
            w.it = 1.0f / zt;
            w.id = 1.0f / zd;
            w.c2 = f2(c, c);
            w.C = 0.0f;
            for (int i = tid; i < nk; i += TTH) {
                const int x = S.tok[S.kids[i]];
                using L = Lg<DT>;
                const float lt = L::load1(P.target, off + x);
                const float ld = L::load1(P.draft, off + x);
                S.r0[i] = (ld == -INFINITY) ? -1.0f
                                            : ex2(((lt - mt) - (ld - md)) * c) * (zd / zt);
            }
            __syncthreads();
            float M = 1.0f, R = 0.0f;
            bool fresh = false;  // S.wtot holds the pass for the current C
            for (int i = 0; i < nk; ++i) {
                const float r0 = S.r0[i];
                if (r0 < 0.0f) {
                    err = true;
                    break;
                }
                const float ratio = fmaxf(0.0f, r0 - w.C) / M;
                const int kid = S.kids[i];
                if (ratio >= 1.0f || P.u_accept[(size_t)b * N + kid] < ratio) {
                    next = kid;
                    break;
                }
                w.C += M;
                M = residual_pass<DT>(P, off, w, S, warp, lane, ring);
                R = M;
                fresh = true;
                if (!(M > 0.0f)) {  // rounding only: draw from p_c
                    w.C = 0.0f;
                    fresh = false;
                    break;
                }
            }
            if (err)
                break;
            if (next < 0) {
                if (!(fresh && R > 0.0f)) {
                    // draw from p_c (a leaf, or the rounding fallback): the
                    // statistics pass's per-warp partials are the segment masses
                    w.C = 0.0f;
                    if (tid < TW)
                        S.wtot[tid] = rescale(S.red_s[tid], S.red_m[tid], mt, c) * w.it;
                    __syncthreads();
                    R = 0.0f;
                    for (int i = 0; i < TW; ++i)
                        R += S.wtot[i];
                }
                if (!(R > 0.0f)) {
                    err = true;
                    break;
                }
                token = draw_from<DT>(P, off, w, R, P.u_resample[b], S, warp, lane);
                break;
            }
        }
        if (tid == 0)
            S.path[depth] = next;
        ++depth;
        cur = next;
        __syncthreads();
    }
    __syncthreads();
    for (int i = tid; i < N; i += TTH) {
        int on = -1, ot = -1;
        if (!err) {
            if (i < depth) {
                on = S.path[i];
                ot = S.tok[on];
            } else if (i == depth) {
                ot = token;
            }
        }
        P.out_nodes[(size_t)b * N + i] = on;
        P.out_tokens[(size_t)b * N + i] = ot;
    }
    if (tid == 0)
        P.out_n[b] = err ? -1 : depth;
}

std::atomic<bool> g_attr[64][2];  // the kernel's shared-memory limit raised, per device and dtype

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace

extern "C" {

int32_t spec_verify_tree(const void *target_logits, const void *draft_logits,
                         const int32_t *parent, const int32_t *tokens, const int32_t *n_nodes,
                         const float *u_accept, const float *u_resample,
                         const float *temperature, int32_t *out_tokens, int32_t *out_nodes,
                         int32_t *out_num_accepted, int32_t B, int32_t N, int32_t V,
                         int32_t dtype, void *stream)
{
    if (B < 0 || N < 1 || N > SPEC_TREE_MAX_NODES || V < 2 || V > SPEC_MAX_V ||
        (dtype != SPEC_F32 && dtype != SPEC_BF16))
        return SPEC_EINVAL;
    if (B == 0)
        return SPEC_OK;
    if (!target_logits || !draft_logits || !parent || !tokens || !n_nodes || !u_accept ||
        !u_resample || !temperature || !out_tokens || !out_nodes || !out_num_accepted)
        return SPEC_EINVAL;
    if (!aligned(target_logits, 16) || !aligned(draft_logits, 16) || !aligned(parent, 4) ||
        !aligned(tokens, 4) || !aligned(n_nodes, 4) || !aligned(u_accept, 4) ||
        !aligned(u_resample, 4) || !aligned(temperature, 4) || !aligned(out_tokens, 4) ||
        !aligned(out_nodes, 4) || !aligned(out_num_accepted, 4))
        return SPEC_EINVAL;
    TParams P;
    P.target = target_logits;
    P.draft = draft_logits;
    P.parent = parent;
    P.tokens = tokens;
    P.n_nodes = n_nodes;
    P.u_accept = u_accept;
    P.u_resample = u_resample;
    P.temperature = temperature;
    P.out_tokens = out_tokens;
    P.out_nodes = out_nodes;
    P.out_n = out_num_accepted;
    P.N = N;
    P.V = V;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the per-thread cp.async slots take the kernel above the 48 KB of shared
    // memory a launch gets by default: raised once per device and dtype
    // (published with release order; racing threads repeat the same call)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SPEC_ECUDA;
    const int di = (dtype == SPEC_F32) ? 0 : 1;
    if (!g_attr[dev][di].load(std::memory_order_acquire)) {
        const void *fn = (dtype == SPEC_F32) ? (const void *)tree_kernel<SPEC_F32>
                                             : (const void *)tree_kernel<SPEC_BF16>;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)RING_BYTES) != cudaSuccess)
            return SPEC_ECUDA;
        g_attr[dev][di].store(true, std::memory_order_release);
    }
    if (dtype == SPEC_F32)
        tree_kernel<SPEC_F32><<<(unsigned int)B, TTH, RING_BYTES, st>>>(P);
    else
        tree_kernel<SPEC_BF16><<<(unsigned int)B, TTH, RING_BYTES, st>>>(P);
    if (cudaPeekAtLastError() != cudaSuccess) {
        (void)cudaGetLastError();
        return SPEC_ECUDA;
    }
    return SPEC_OK;
}

}  // extern "C"
