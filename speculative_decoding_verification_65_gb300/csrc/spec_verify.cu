// spec_verify.cu -- GB300 (sm_103a) kernel and C ABI for batched
// speculative-sampling verification.
//
// The operation is the verification step of speculative decoding as stated in
// "Speculative Decoding and the Art of Fast LLM Inference" ("The Algorithm,
// Step by Step"), the thelatentsource article "speculative-decoding-llm-speed"
// ("The correction that keeps the target in charge": the accept_token snippet
// and the residual r(x)) and the techaiinterview answer "How does speculative
// decoding work, why is it lossless, and how much does it speed things up?"
// ("Algorithm (one round)"; greedy remark in "Deep dive").
//
// Design: one persistent, warp-specialised kernel per call.
//   * Work unit = tile: a 32 KB segment of one logits row (a target or draft
//     position of one sequence).  Tiles are numbered sequence-major and handed
//     out by a global atomic counter.
//   * Each CTA has three roles and no CTA-wide barrier after start-up:
//       - producer warp: claims tiles and moves them with cp.async.bulk (the
//         TMA bulk-copy engine) into a 3-stage shared-memory ring guarded by
//         mbarriers; it also injects "draw tiles" when the sequencer asks;
//       - 8 consumer warps: per tile, each warp reduces its share to a partial
//         (row maximum m, lowest-index argmax, Z = sum 2^((x-m)*log2(e)/T))
//         and the last warp to finish combines the 8 partials into the tile's
//         16-byte partial in the workspace; for a draw tile each warp writes
//         inverse-CDF chunk totals instead;
//       - sequencer warp: counts finished tiles per sequence with one atomic
//         ticket per tile; the CTA that completes a sequence combines its row
//         statistics, runs the accept scan (first rejection), asks the
//         producer to stream the one or two rows the correction / bonus draw
//         needs (still L2-resident) as draw tiles, and finally locates the
//         token inside one 32-lane chunk.
//   * Reduction orders depend only on row-relative indices, never on which
//     CTA or warp handled a tile or on the row's address, so bit-identical
//     target and draft rows give bit-identical statistics (ratio exactly 1).
//   * Every wait is bounded: a timed-out wait records SPEC_DEV_WAIT_TIMEOUT in
//     the workspace and the kernel returns; nothing traps.
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "spec_verify.h"

namespace {

constexpr int NCW = 8;                           // consumer warps
constexpr int NT = NCW * 32;                     // consumer threads
constexpr int WARP_P = NCW;                      // producer warp
constexpr int WARP_S = NCW + 1;                  // sequencer warp
constexpr int NTHREADS = (NCW + 2) * 32;
constexpr int STAGES = 3;                        // shared-memory ring depth
constexpr int TILE_BYTES = 32768;                // one stats tile of one row
constexpr int HALF_BYTES = TILE_BYTES / 2;       // one row's share of a draw tile
constexpr int SLOT_BYTES = TILE_BYTES + 128;     // room for misaligned heads/tails
constexpr int HALF_OFFSET = HALF_BYTES + 64;     // draft half of a draw slot
constexpr int U = TILE_BYTES / (NT * 16);        // 16-byte vectors per consumer per stats tile
constexpr int UD = HALF_BYTES / (NT * 16);       // CDF blocks per draw tile
constexpr int MAX_ROWS = 2 * SPEC_MAX_K + 1;
constexpr int MAXBLK = SPEC_MAX_V / (NT * 4) + UD;  // CDF blocks per row, worst case
constexpr int EVQ = 64;                          // consumer -> sequencer events
constexpr int RQ = 8;                            // sequencer -> producer draw requests
constexpr int NJ = 4;                            // draw jobs in flight per CTA
constexpr int PEND = 64;                         // completed sequences awaiting a scan
constexpr int BACKLOG = 16;                      // producer pauses stats tiles above this
constexpr float LOG2E = 1.4426950408889634f;
constexpr unsigned long long WAIT_NS = 2000000000ull;  // 2 s bound on any wait

static_assert(U * NT * 16 == TILE_BYTES, "stats tile must split evenly over consumers");
static_assert(UD * NT * 16 == HALF_BYTES, "draw tile must split evenly over consumers");
static_assert(RQ >= NJ, "every job can be requested at once");

struct WsHeader {
    unsigned int tile_counter;
    unsigned int ctas_done;
    int status;
    unsigned int pad[61];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

enum { KIND_END = 0, KIND_STATS = 1, KIND_DRAW = 2 };
enum { MODE_SKIP = 0, MODE_GREEDY = 1, MODE_SAMPLE = 2 };   // stats tiles
enum { DRAW_RESIDUAL = 1, DRAW_TARGET = 2 };                // draw tiles / jobs

struct TileInfo {
    int kind;
    int b;         // sequence
    int rsq;       // stats: row in sequence (0..k target, k+1..2k draft)
    int seg;       // stats: tile of the row; draw: draw tile of the row
    int mode;
    int job;       // draw: job slot
    float c;       // stats: log2(e) / T
    int phase0;    // bytes from the copy start to the first element (target / stats row)
    int ncopied0;  // bytes present in the slot
    int phase1;    // the same for the draft half of a draw tile
    int ncopied1;
    int pad;
};

struct Job {
    int state;     // 0 free, 1 drawing, 2 chunk totals complete
    int b, j, mode, nseg, done;
    int pad0, pad1;
    long long t_row, d_row;
    float mt, rzt, md, rzd, c, u;
};

struct Params {
    const void *target;
    const void *draft;
    const int32_t *tokens;
    const float *u_accept;
    const float *u_resample;
    const float *temperature;
    int32_t *out_tokens;
    int32_t *out_num_accepted;
    float *out_probs;  // nullable
    uint8_t *ws;
    unsigned int *seq_count;
    float4 *part;
    float *chunks;
    int B, k, V;
    int NS;            // stats tiles per row
    int rows;          // rows per sequence (2k+1)
    int DS;            // draw tiles per row
    int chunk_stride;  // floats of chunk totals per sequence
    unsigned int total_tiles;
    unsigned long long target_bytes, draft_bytes;
};

struct Smem {
    unsigned long long full[STAGES];
    unsigned long long empty[STAGES];
    TileInfo info[STAGES];
    float4 wpart[STAGES][NCW];
    int wcnt[STAGES];
    int ev_w, ev_r;
    int evq[EVQ];
    int ev_seq[EVQ];
    int rq[RQ];
    int rq_w;
    int drain, stats_issued, finish, abort, backlog;
    int pend[PEND];
    Job jobs[NJ];
    float rm[MAX_ROWS], rZ[MAX_ROWS];
    int rarg[MAX_ROWS], rbad[MAX_ROWS];
    float btot[MAXBLK];
};

constexpr size_t SMEM_BYTES = (size_t)STAGES * SLOT_BYTES + sizeof(Smem);

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

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (globaltimer() - t0 > WAIT_NS)
            return false;
    }
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
// same result).  The order depends only on lane numbers.
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
    }
    int cand = (m == mw) ? idx : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
    m = mw;
    idx = cand;
}


__device__ __forceinline__ int vld(const int &x) { return *reinterpret_cast<const volatile int *>(&x); }
__device__ __forceinline__ void vst(int &x, int v) { *reinterpret_cast<volatile int *>(&x) = v; }

__device__ __forceinline__ void raise_abort(Smem &S, WsHeader *hdr)
{
    atomicExch(&hdr->status, SPEC_DEV_WAIT_TIMEOUT);
    vst(S.abort, 1);
}

__device__ __forceinline__ bool temperature_valid(float T)
{
    return !(isnan(T) || T < 0.0f || isinf(T) || (T > 0.0f && T < FLT_MIN));
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
    int e0, e1, phase, ncopied;
    bool fast;
};

template <int DT>
__device__ __forceinline__ Seg make_seg(const Params &P, const uint8_t *slot, const void *arr,
                                        size_t row, int e0, int e1, int phase, int ncopied)
{
    using L = Lg<DT>;
    Seg g;
    g.slot = slot;
    g.arr = arr;
    g.row = row;
    g.e0 = e0;
    g.e1 = e1;
    g.phase = phase;
    g.ncopied = ncopied;
    const int nbytes = (e1 - e0) * L::ES;
    g.fast = (phase == 0) && ((nbytes & 15) == 0) && (ncopied >= nbytes);
    return g;
}

template <int DT>
__device__ __forceinline__ uint4 seg_vec(const Params &P, const Seg &g, int v)
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
                bits = __float_as_uint(L::load1(g.arr, g.row * (size_t)P.V + e)) >> (DT == SPEC_BF16 ? 16 : 0);
            L::put(r, j, bits);
        }
    }
    return r;
}

// Row vector straight from global memory (L2), for the final chunk search.
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

// ----------------------------------------------------------- stats tiles

// Per-thread statistics of one stats tile: consumer thread t owns vectors
// t, t+NT, ... of the tile.  Maximum over the registers first, then exactly
// one exponential per element.
template <int DT>
__device__ __forceinline__ void tile_thread_stats(const Params &P, const Seg &g, int tid,
                                                  int mode, float c, float &m_out,
                                                  float &s_out, int &idx_out)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    const int v0 = g.e0 / VEC;
    const int v1 = (g.e1 + VEC - 1) / VEC;

    uint4 raw[U];
    float vmax[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int v = v0 + tid + u * NT;
        raw[u] = (v < v1) ? seg_vec<DT>(P, g, v) : neg_inf_vec(L::NEG_INF_WORD);
        float x[VEC];
        L::unpack(raw[u], x);
        float a = fmax_nan(x[0], x[1]);
#pragma unroll
        for (int j = 2; j < VEC; j += 2)
            a = fmax_nan(a, fmax_nan(x[j], x[j + 1]));
        vmax[u] = a;
    }
    float m = vmax[0];
#pragma unroll
    for (int u = 1; u < U; ++u)
        m = fmax_nan(m, vmax[u]);

    int idx = INT_MAX;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (idx == INT_MAX && vmax[u] == m && (v0 + tid + u * NT) < v1) {
            float x[VEC];
            L::unpack(raw[u], x);
#pragma unroll
            for (int j = VEC - 1; j >= 0; --j)
                if (x[j] == m)
                    idx = (v0 + tid + u * NT) * VEC + j;
        }
    }

    float s = 0.0f;
    if (mode == MODE_SAMPLE && m != -INFINITY) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float x[VEC];
            L::unpack(raw[u], x);
            float sv[VEC];
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                sv[j] = ex2((x[j] - m) * c);
#pragma unroll
            for (int w = VEC / 2; w > 0; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j)
                    sv[j] = sv[j] + sv[j + w];
            s += sv[0];
        }
    }
    m_out = m;
    s_out = s;
    idx_out = idx;
}

// ------------------------------------------------------------ draw weights
//
// w(x) = max(0, p(x) - q(x)) (residual) or the unnormalised target weight
// 2^((t(x)-m)*c) (bonus, or the rounding-only fallback).  -inf padding gives 0.

template <int DT>
__device__ __forceinline__ void draw_weights(const Job &J, const uint4 &rt, const uint4 &rd,
                                             float (&w)[Lg<DT>::VEC])
{
    using L = Lg<DT>;
    float xt[L::VEC];
    L::unpack(rt, xt);
    if (J.mode == DRAW_RESIDUAL) {
        float xd[L::VEC];
        L::unpack(rd, xd);
#pragma unroll
        for (int j = 0; j < L::VEC; ++j) {
            const float p = ex2((xt[j] - J.mt) * J.c) * J.rzt;
            const float q = ex2((xd[j] - J.md) * J.c) * J.rzd;
            w[j] = fmaxf(p - q, 0.0f);
        }
    } else {
#pragma unroll
        for (int j = 0; j < L::VEC; ++j)
            w[j] = ex2((xt[j] - J.mt) * J.c);
    }
}

// Inclusive Kogge-Stone scan of one value per lane, and its exclusive shift.
__device__ __forceinline__ void warp_scan(float tau, int lane, float &incl, float &excl)
{
    float x = tau;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x = x + y;
    }
    incl = x;
    const float e = __shfl_up_sync(0xffffffffu, x, 1);
    excl = (lane == 0) ? 0.0f : e;
}

// The inverse CDF's running mass C(x) is defined by a fixed hierarchy:
//   element -> lane (VEC elements, left to right) -> chunk (32 lanes,
//   Kogge-Stone) -> block (8 chunks, left to right) -> row (blocks, left to
//   right).  A block is NT vectors; chunk w of block k holds vectors
//   k*NT + 32*w .. k*NT + 32*w + 31.  A draw tile holds UD blocks.
// Consumer warp `warp` writes the totals of chunk `warp` of each block.
template <int DT>
__device__ __forceinline__ void draw_tile_chunks(const Params &P, const TileInfo &ti,
                                                 const Job &J, const uint8_t *slot, int warp,
                                                 int lane)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    constexpr int DSEG = HALF_BYTES / L::ES;
    const int e0 = ti.seg * DSEG;
    const int e1 = min(P.V, e0 + DSEG);
    const Seg gt = make_seg<DT>(P, slot, P.target, (size_t)J.t_row, e0, e1, ti.phase0, ti.ncopied0);
    const Seg gd = make_seg<DT>(P, slot + HALF_OFFSET, P.draft, (size_t)J.d_row, e0, e1,
                                ti.phase1, ti.ncopied1);
    float *out = P.chunks + (size_t)J.b * P.chunk_stride + (size_t)ti.seg * UD * NCW;
#pragma unroll
    for (int u = 0; u < UD; ++u) {
        const int v = e0 / VEC + u * NT + warp * 32 + lane;
        const uint4 rt = seg_vec<DT>(P, gt, v);
        const uint4 rd = (J.mode == DRAW_RESIDUAL) ? seg_vec<DT>(P, gd, v) : rt;
        float w[VEC];
        draw_weights<DT>(J, rt, rd, w);
        float tau = 0.0f;
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            tau = tau + w[j];
        float incl, excl;
        warp_scan(tau, lane, incl, excl);
        if (lane == 31)
            __stcg(out + u * NCW + warp, incl);
    }
}

// ------------------------------------------------------------- sequencer

// Row statistics and the accept scan for a completed sequence (sequencer
// warp).  Greedy and error sequences get their outputs here; a sampling
// sequence gets draw job `jb` (posted to the producer).
template <int DT>
__device__ void sequence_scan(const Params &P, Smem &S, int b, int jb, int lane)
{
    using L = Lg<DT>;
    const int k = P.k, V = P.V;
    const float T = __ldg(P.temperature + b);
    const bool tvalid = temperature_valid(T);
    const bool greedy = tvalid && T == 0.0f;
    const float c = (tvalid && !greedy) ? LOG2E / T : 0.0f;

    // 1. fold each row's tile partials left to right (one lane per row)
    const int nrows = tvalid ? (greedy ? k + 1 : P.rows) : 0;
    for (int r = lane; r < nrows; r += 32) {
        float m = -INFINITY, s = 0.0f;
        int idx = INT_MAX;
        float4 *pp = P.part + ((size_t)b * P.rows + r) * P.NS;
        for (int sg0 = 0; sg0 < P.NS; sg0 += 4) {
            float4 pv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                pv[q] = (sg0 + q < P.NS) ? __ldcg(pp + sg0 + q) : make_float4(-INFINITY, 0.0f, __int_as_float(INT_MAX), 0.0f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (sg0 + q < P.NS) {
                    __stcg(pp + sg0 + q, make_float4(0.0f, 0.0f, 0.0f, 0.0f));
                    const float pm = pv[q].x, ps = pv[q].y;
                    const int pi = __float_as_int(pv[q].z);
                    const float mn = fmax_nan(m, pm);
                    if (!greedy)
                        s = rescale(s, m, mn, c) + rescale(ps, pm, mn, c);
                    idx = (m == mn && pm == mn) ? min(idx, pi) : (pm == mn ? pi : idx);
                    m = mn;
                }
            }
        }
        S.rm[r] = m;
        S.rZ[r] = s;
        S.rarg[r] = idx;
        S.rbad[r] = (isnan(m) || isinf(m)) ? 1 : 0;  // NaN, +inf, or all -inf
    }
    __syncwarp();

    // 2. accept scan: lane i tests position i
    bool err = !tvalid;
    int g = 0;
    bool fail = false, qzero = false;
    if (!err) {
        if (lane < k) {
            g = __ldg(P.tokens + (size_t)b * k + lane);
            if (g < 0 || g >= V)
                err = true;
        }
        for (int r = lane; r < nrows; r += 32)
            if (S.rbad[r])
                err = true;
        err = __any_sync(0xffffffffu, err);
    }
    int j = k, token = -1;
    if (!err) {
        if (greedy) {
            fail = (lane < k) && (g != S.rarg[lane]);
        } else if (lane < k) {
            const size_t rt = (size_t)b * (k + 1) + lane, rd = (size_t)b * k + lane;
            const float lt = L::load1(P.target, rt * V + g);
            const float ld = L::load1(P.draft, rd * V + g);
            const float mt = S.rm[lane], zt = S.rZ[lane];
            const float md = S.rm[k + 1 + lane], zd = S.rZ[k + 1 + lane];
            qzero = (ld == -INFINITY);
            const float dt = lt - mt, dd = ld - md;
            const float x = (dt - dd) * c;
            const float ratio = ((x == 0.0f) ? 1.0f : ex2(x)) * (zd / zt);
            const float ua = __ldg(P.u_accept + (size_t)b * k + lane);
            fail = qzero || !((ratio >= 1.0f) || (ua < ratio));
            if (P.out_probs) {
                P.out_probs[((size_t)b * k + lane) * 2 + 0] = ex2(dt * c) / zt;
                P.out_probs[((size_t)b * k + lane) * 2 + 1] = ex2(dd * c) / zd;
            }
        }
        const unsigned fm = __ballot_sync(0xffffffffu, fail);
        j = fm ? (__ffs(fm) - 1) : k;
        if (!greedy) {
            const unsigned qm = __ballot_sync(0xffffffffu, qzero);
            if (j < k && ((qm >> j) & 1u))
                err = true;
        } else {
            token = S.rarg[j];
        }
    }
    if (P.out_probs && (err || greedy) && lane < k) {
        P.out_probs[((size_t)b * k + lane) * 2 + 0] = __int_as_float(0x7fc00000);
        P.out_probs[((size_t)b * k + lane) * 2 + 1] = __int_as_float(0x7fc00000);
    }

    if (err || greedy) {
        for (int i = lane; i <= k; i += 32) {
            int o = -1;
            if (!err)
                o = (i < j) ? __ldg(P.tokens + (size_t)b * k + i) : (i == j ? token : -1);
            P.out_tokens[(size_t)b * (k + 1) + i] = o;
        }
        if (lane == 0) {
            P.out_num_accepted[b] = err ? -1 : j;
            atomicExch(P.seq_count + b, 0u);
        }
        __syncwarp();
        return;
    }

    // 3. a draw job: the residual at the rejected position, or the bonus row
    if (lane == 0) {
        Job &J = S.jobs[jb];
        J.b = b;
        J.j = j;
        J.c = c;
        J.t_row = (long long)b * (k + 1) + j;
        J.mt = S.rm[j];
        J.rzt = 1.0f / S.rZ[j];
        if (j < k) {
            J.mode = DRAW_RESIDUAL;
            J.d_row = (long long)b * k + j;
            J.md = S.rm[k + 1 + j];
            J.rzd = 1.0f / S.rZ[k + 1 + j];
        } else {
            J.mode = DRAW_TARGET;
            J.d_row = J.t_row;
            J.md = J.mt;
            J.rzd = J.rzt;
        }
        J.u = __ldg(P.u_resample + b);
        J.nseg = P.DS;
        J.done = 0;
        vst(J.state, 1);
        __threadfence_block();
        S.rq[S.rq_w % RQ] = jb;
        __threadfence_block();
        vst(S.rq_w, S.rq_w + 1);
    }
    __syncwarp();
}

// Locate the drawn token once every chunk total of job jb is known
// (sequencer warp): block by block, then chunk by chunk, then within the
// chunk, C(x) = base + (W + (E + s)) with base the running block sum, W the
// running chunk sum in the block, E the lane's exclusive scan and s the
// lane's running sum.  The token is the smallest x with w(x) > 0 and
// C(x) > u * R, R the row total; if rounding leaves none in the chunk found,
// the chunk's last positive-weight token.
template <int DT>
__device__ void final_search(const Params &P, Smem &S, int jb, int lane)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    const Job J = S.jobs[jb];
    const int k = P.k;
    const int nblk = J.nseg * UD;
    float *ch = P.chunks + (size_t)J.b * P.chunk_stride;

    for (int blk = lane; blk < nblk; blk += 32) {
        float c8[NCW];
#pragma unroll
        for (int w = 0; w < NCW; ++w)
            c8[w] = __ldcg(ch + blk * NCW + w);
        float bt = 0.0f;
#pragma unroll
        for (int w = 0; w < NCW; ++w)
            bt = bt + c8[w];
        S.btot[blk] = bt;
    }
    __syncwarp();
    float R = 0.0f, uR = 0.0f, base = 0.0f;
    int bstar = 0, wstar = NCW - 1;
    float Wst = 0.0f;
    if (lane == 0) {
        for (int blk = 0; blk < nblk; ++blk)
            R = R + S.btot[blk];
        uR = J.u * R;
        float acc = 0.0f;
        bstar = nblk - 1;
        for (int blk = 0; blk < nblk; ++blk) {
            const float nxt = acc + S.btot[blk];
            if (nxt > uR) {
                bstar = blk;
                break;
            }
            acc = nxt;
        }
        base = acc;
        if (R > 0.0f) {
            float W = 0.0f;
            for (int w = 0; w < NCW; ++w) {
                const float nxt = W + __ldcg(ch + bstar * NCW + w);
                if (base + nxt > uR) {
                    wstar = w;
                    break;
                }
                W = nxt;
            }
            Wst = W;
        }
    }
    R = __shfl_sync(0xffffffffu, R, 0);
    uR = __shfl_sync(0xffffffffu, uR, 0);
    base = __shfl_sync(0xffffffffu, base, 0);
    Wst = __shfl_sync(0xffffffffu, Wst, 0);
    bstar = __shfl_sync(0xffffffffu, bstar, 0);
    wstar = __shfl_sync(0xffffffffu, wstar, 0);

    if (!(R > 0.0f)) {
        if (J.mode == DRAW_RESIDUAL) {
            // the residual vanished by rounding alone: draw from p_j instead
            if (lane == 0) {
                Job &Jm = S.jobs[jb];
                Jm.mode = DRAW_TARGET;
                Jm.d_row = Jm.t_row;
                Jm.md = Jm.mt;
                Jm.rzd = Jm.rzt;
                Jm.done = 0;
                vst(Jm.state, 1);
                __threadfence_block();
                S.rq[S.rq_w % RQ] = jb;
                __threadfence_block();
                vst(S.rq_w, S.rq_w + 1);
            }
            __syncwarp();
            return;
        }
    }

    int tok = -1;
    if (R > 0.0f) {
        const int v = bstar * NT + wstar * 32 + lane;
        const uint4 rt = row_vec<DT>(P.target, (size_t)J.t_row, v, P.V);
        const uint4 rd = (J.mode == DRAW_RESIDUAL) ? row_vec<DT>(P.draft, (size_t)J.d_row, v, P.V) : rt;
        float w[VEC];
        draw_weights<DT>(J, rt, rd, w);
        float sacc[VEC];
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            s = s + w[j];
            sacc[j] = s;
        }
        float incl, excl;
        warp_scan(s, lane, incl, excl);
        const float pre = Wst + excl;
        int cand = INT_MAX, lastp = -1;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const int e = v * VEC + j;
            if (w[j] > 0.0f) {
                lastp = e;
                if (cand == INT_MAX && base + (pre + sacc[j]) > uR)
                    cand = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
            lastp = max(lastp, __shfl_xor_sync(0xffffffffu, lastp, o));
        }
        tok = (cand != INT_MAX) ? cand : lastp;
    }

    const bool err = tok < 0;
    const int b = J.b;
    for (int i = lane; i <= k; i += 32) {
        int o = -1;
        if (!err)
            o = (i < J.j) ? __ldg(P.tokens + (size_t)b * k + i) : (i == J.j ? tok : -1);
        P.out_tokens[(size_t)b * (k + 1) + i] = o;
    }
    // leave the chunk totals zeroed for the next call
    for (int i = lane; i < nblk * NCW; i += 32)
        __stcg(ch + i, 0.0f);
    __syncwarp();
    if (lane == 0) {
        P.out_num_accepted[b] = err ? -1 : J.j;
        atomicExch(P.seq_count + b, 0u);
        vst(S.jobs[jb].state, 0);
    }
    __syncwarp();
}

// ------------------------------------------------------------------ kernel

template <int DT>
__global__ void __launch_bounds__(NTHREADS, 2) spec_verify_kernel(const Params P)
{
    using L = Lg<DT>;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *slots = smem_raw;
    Smem &S = *reinterpret_cast<Smem *>(smem_raw + (size_t)STAGES * SLOT_BYTES);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(P.ws);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const unsigned int tiles_per_seq = (unsigned int)P.rows * (unsigned int)P.NS;
    constexpr int SEG = TILE_BYTES / L::ES;
    constexpr int DSEG = HALF_BYTES / L::ES;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], NCW);
            S.wcnt[s] = 0;
        }
        S.ev_w = 0;
        S.ev_r = 0;
        for (int i = 0; i < EVQ; ++i)
            S.ev_seq[i] = 0;
        S.rq_w = 0;
        S.drain = 0;
        S.stats_issued = 0;
        S.finish = 0;
        S.abort = 0;
        S.backlog = 0;
        for (int i = 0; i < NJ; ++i)
            S.jobs[i].state = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    if (warp == WARP_P) {
        // ------------------------------------------------------- producer
        if (lane != 0)
            return;
        int stage = 0;
        uint32_t phase = 0;
        int issued_phase[STAGES];
        for (int s = 0; s < STAGES; ++s)
            issued_phase[s] = -1;
        int rq_r = 0;
        int stats_issued = 0;
        bool drained = false;
        unsigned long long idle_t0 = globaltimer();
        unsigned int t = atomicAdd(&hdr->tile_counter, 1u);
        bool ok = true;

        auto acquire = [&]() -> bool {
            if (!mbar_wait(&S.empty[stage], phase ^ 1u)) {
                raise_abort(S, hdr);
                return false;
            }
            return true;
        };
        auto advance = [&]() {
            issued_phase[stage] = (int)phase;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        };
        // copy the aligned byte range around elements [e0, e1) of `row` into `dst`
        auto copy_seg = [&](const uint8_t *arr, unsigned long long arr_bytes, size_t row, int e0,
                            int e1, uint8_t *dst, int &ph, int &nc) -> uint32_t {
            const unsigned long long start = ((unsigned long long)row * P.V + e0) * L::ES;
            const unsigned long long end = ((unsigned long long)row * P.V + e1) * L::ES;
            const unsigned long long a0 = start & ~15ull;
            unsigned long long a1 = (end + 15) & ~15ull;
            const unsigned long long lim = arr_bytes & ~15ull;
            if (a1 > lim)
                a1 = lim;
            ph = (int)(start - a0);
            const uint32_t bytes = (a1 > a0) ? (uint32_t)(a1 - a0) : 0u;
            nc = (int)bytes;
            if (bytes)
                bulk_copy_g2s(dst, arr + a0, bytes, &S.full[stage]);
            return bytes;
        };

        while (ok) {
            if (vld(S.abort))
                break;
            // a draw request first: its rows are L2-resident right now
            if (vld(S.rq_w) != rq_r) {
                __threadfence_block();
                const int jb = S.rq[rq_r % RQ];
                ++rq_r;
                const Job J = S.jobs[jb];
                for (int sg = 0; sg < J.nseg && ok; ++sg) {
                    if (!(ok = acquire()))
                        break;
                    TileInfo &ti = S.info[stage];
                    ti.kind = KIND_DRAW;
                    ti.b = J.b;
                    ti.seg = sg;
                    ti.mode = J.mode;
                    ti.job = jb;
                    const int e0 = sg * DSEG, e1 = min(P.V, e0 + DSEG);
                    uint8_t *dst = slots + (size_t)stage * SLOT_BYTES;
                    uint32_t bytes = 0;
                    // the transaction count must be armed before any copy can land
                    const unsigned long long st0 = ((unsigned long long)J.t_row * P.V + e0) * L::ES;
                    const unsigned long long en0 = ((unsigned long long)J.t_row * P.V + e1) * L::ES;
                    unsigned long long a0 = st0 & ~15ull, a1 = (en0 + 15) & ~15ull;
                    if (a1 > (P.target_bytes & ~15ull)) a1 = P.target_bytes & ~15ull;
                    uint32_t expect = (a1 > a0) ? (uint32_t)(a1 - a0) : 0u;
                    if (J.mode == DRAW_RESIDUAL) {
                        const unsigned long long st1 = ((unsigned long long)J.d_row * P.V + e0) * L::ES;
                        const unsigned long long en1 = ((unsigned long long)J.d_row * P.V + e1) * L::ES;
                        unsigned long long b0 = st1 & ~15ull, b1 = (en1 + 15) & ~15ull;
                        if (b1 > (P.draft_bytes & ~15ull)) b1 = P.draft_bytes & ~15ull;
                        expect += (b1 > b0) ? (uint32_t)(b1 - b0) : 0u;
                    }
                    if (expect)
                        mbar_arrive_expect_tx(&S.full[stage], expect);
                    bytes += copy_seg(reinterpret_cast<const uint8_t *>(P.target), P.target_bytes,
                                      (size_t)J.t_row, e0, e1, dst, ti.phase0, ti.ncopied0);
                    if (J.mode == DRAW_RESIDUAL) {
                        bytes += copy_seg(reinterpret_cast<const uint8_t *>(P.draft), P.draft_bytes,
                                          (size_t)J.d_row, e0, e1, dst + HALF_OFFSET, ti.phase1,
                                          ti.ncopied1);
                    } else {
                        ti.phase1 = 0;
                        ti.ncopied1 = 0;
                    }
                    if (!expect)
                        mbar_arrive(&S.full[stage]);
                    advance();
                }
                idle_t0 = globaltimer();
                continue;
            }
            if (t < P.total_tiles && vld(S.backlog) < BACKLOG) {
                if (!(ok = acquire()))
                    break;
                const int b = (int)(t / tiles_per_seq);
                const unsigned int rem = t - (unsigned int)b * tiles_per_seq;
                const int rsq = (int)(rem / (unsigned int)P.NS);
                const int seg = (int)(rem - (unsigned int)rsq * (unsigned int)P.NS);
                const float T = __ldg(P.temperature + b);
                int mode;
                if (!temperature_valid(T))
                    mode = MODE_SKIP;
                else if (T == 0.0f)
                    mode = (rsq <= P.k) ? MODE_GREEDY : MODE_SKIP;  // greedy never reads drafts
                else
                    mode = MODE_SAMPLE;
                TileInfo &ti = S.info[stage];
                ti.kind = KIND_STATS;
                ti.b = b;
                ti.rsq = rsq;
                ti.seg = seg;
                ti.mode = mode;
                ti.c = (mode == MODE_SAMPLE) ? LOG2E / T : 0.0f;
                ti.phase1 = 0;
                ti.ncopied1 = 0;
                uint32_t bytes = 0;
                if (mode != MODE_SKIP) {
                    const bool is_target = rsq <= P.k;
                    const uint8_t *arr = reinterpret_cast<const uint8_t *>(is_target ? P.target : P.draft);
                    const unsigned long long arr_bytes = is_target ? P.target_bytes : P.draft_bytes;
                    const size_t row = is_target ? (size_t)b * (P.k + 1) + rsq
                                                 : (size_t)b * P.k + (rsq - P.k - 1);
                    const int e0 = seg * SEG, e1 = min(P.V, e0 + SEG);
                    const unsigned long long st0 = ((unsigned long long)row * P.V + e0) * L::ES;
                    const unsigned long long en0 = ((unsigned long long)row * P.V + e1) * L::ES;
                    unsigned long long a0 = st0 & ~15ull, a1 = (en0 + 15) & ~15ull;
                    if (a1 > (arr_bytes & ~15ull)) a1 = arr_bytes & ~15ull;
                    const uint32_t expect = (a1 > a0) ? (uint32_t)(a1 - a0) : 0u;
                    if (expect)
                        mbar_arrive_expect_tx(&S.full[stage], expect);
                    bytes = copy_seg(arr, arr_bytes, row, e0, e1, slots + (size_t)stage * SLOT_BYTES,
                                     ti.phase0, ti.ncopied0);
                } else {
                    ti.phase0 = 0;
                    ti.ncopied0 = 0;
                }
                if (!bytes)
                    mbar_arrive(&S.full[stage]);
                ++stats_issued;
                advance();
                t = atomicAdd(&hdr->tile_counter, 1u);
                idle_t0 = globaltimer();
                continue;
            }
            if (t >= P.total_tiles && !drained) {
                vst(S.stats_issued, stats_issued);
                __threadfence_block();
                vst(S.drain, 1);
                drained = true;
            }
            if (drained && vld(S.finish)) {
                if (!(ok = acquire()))
                    break;
                S.info[stage].kind = KIND_END;
                mbar_arrive(&S.full[stage]);
                advance();
                break;
            }
            if (globaltimer() - idle_t0 > WAIT_NS) {
                raise_abort(S, hdr);
                break;
            }
            __nanosleep(64);
        }
        if (!ok || vld(S.abort)) {
            // let the copies already issued land before leaving
            for (int s = 0; s < STAGES; ++s)
                if (issued_phase[s] >= 0)
                    (void)mbar_wait(&S.full[s], (uint32_t)issued_phase[s]);
        }
        return;
    }

    if (warp < NCW) {
        // ------------------------------------------------------ consumers
        int stage = 0;
        uint32_t phase = 0;
        while (true) {
            if (!mbar_wait(&S.full[stage], phase)) {
                if (lane == 0)
                    raise_abort(S, hdr);
                break;
            }
            const TileInfo ti = S.info[stage];
            if (ti.kind == KIND_END)
                break;
            const uint8_t *slot = slots + (size_t)stage * SLOT_BYTES;
            if (ti.kind == KIND_STATS) {
                float m = -INFINITY, s = 0.0f;
                int idx = INT_MAX;
                if (ti.mode != MODE_SKIP) {
                    const bool is_target = ti.rsq <= P.k;
                    const size_t row = is_target ? (size_t)ti.b * (P.k + 1) + ti.rsq
                                                 : (size_t)ti.b * P.k + (ti.rsq - P.k - 1);
                    const int e0 = ti.seg * SEG, e1 = min(P.V, e0 + SEG);
                    const Seg g = make_seg<DT>(P, slot, is_target ? P.target : P.draft, row, e0, e1,
                                               ti.phase0, ti.ncopied0);
                    tile_thread_stats<DT>(P, g, tid, ti.mode, ti.c, m, s, idx);
                    warp_combine(m, s, idx, ti.c, ti.mode == MODE_SAMPLE);
                }
                if (lane == 0)
                    S.wpart[stage][warp] = make_float4(m, s, __int_as_float(idx), 0.0f);
            } else {
                draw_tile_chunks<DT>(P, ti, S.jobs[ti.job], slot, warp, lane);
            }
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                last = (atomicAdd_block(&S.wcnt[stage], 1) == NCW - 1) ? 1 : 0;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence_block();
                if (ti.kind == KIND_STATS) {
                    if (ti.mode != MODE_SKIP) {
                        float m2 = -INFINITY, s2 = 0.0f;
                        int i2 = INT_MAX;
                        if (lane < NCW) {
                            const float4 r = S.wpart[stage][lane];
                            m2 = r.x;
                            s2 = r.y;
                            i2 = __float_as_int(r.z);
                        }
                        warp_combine(m2, s2, i2, ti.c, ti.mode == MODE_SAMPLE);
                        if (lane == 0)
                            __stcg(P.part + ((size_t)ti.b * P.rows + ti.rsq) * P.NS + ti.seg,
                                   make_float4(m2, s2, __int_as_float(i2), 0.0f));
                    }
                    if (lane == 0) {
                        // hand the finished tile to the sequencer
                        const int et = atomicAdd_block(&S.ev_w, 1);
                        const unsigned long long w0 = globaltimer();
                        bool okq = true;
                        while (et - vld(S.ev_r) >= EVQ) {
                            if (vld(S.abort) || globaltimer() - w0 > WAIT_NS) {
                                raise_abort(S, hdr);
                                okq = false;
                                break;
                            }
                            __nanosleep(32);
                        }
                        if (okq) {
                            S.evq[et % EVQ] = ti.b;
                            __threadfence_block();
                            vst(S.ev_seq[et % EVQ], et + 1);
                        }
                    }
                } else if (lane == 0) {
                    Job &J = S.jobs[ti.job];
                    if (atomicAdd_block(&J.done, 1) == J.nseg - 1) {
                        __threadfence_block();
                        vst(J.state, 2);
                    }
                }
                if (lane == 0)
                    S.wcnt[stage] = 0;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&S.empty[stage]);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        return;
    }

    // ---------------------------------------------------------- sequencer
    if (warp != WARP_S)
        return;
    int pend_r = 0, pend_w = 0;
    unsigned long long last_progress = globaltimer();
    while (true) {
        bool progress = false;
        if (vld(S.abort))
            break;
        // 1. tickets for finished tiles, up to 32 per round
        const int r = S.ev_r;
        const int slot = (r + lane) % EVQ;
        const bool avail = vld(S.ev_seq[slot]) == r + lane + 1;
        const unsigned am = __ballot_sync(0xffffffffu, avail);
        const int nav = (am == 0xffffffffu) ? 32 : (__ffs(~am) - 1);
        if (nav > 0) {
            __threadfence_block();
            int b = -1;
            if (lane < nav)
                b = S.evq[slot];
            __syncwarp();
            if (lane == 0)
                vst(S.ev_r, r + nav);
            bool last = false;
            if (lane < nav) {
                __threadfence();
                last = atomicAdd(P.seq_count + b, 1u) == tiles_per_seq - 1;
            }
            unsigned lm = __ballot_sync(0xffffffffu, last);
            while (lm) {
                const int l = __ffs(lm) - 1;
                lm &= lm - 1;
                const int bb = __shfl_sync(0xffffffffu, b, l);
                if (pend_w - pend_r >= PEND) {
                    if (lane == 0)
                        raise_abort(S, hdr);
                    break;
                }
                if (lane == 0)
                    S.pend[pend_w % PEND] = bb;
                ++pend_w;
            }
            progress = true;
        }
        // 2. draws whose chunk totals are complete
        for (int jb = 0; jb < NJ; ++jb) {
            if (vld(S.jobs[jb].state) == 2) {
                __threadfence_block();
                final_search<DT>(P, S, jb, lane);
                progress = true;
            }
        }
        // 3. completed sequences: row statistics, accept scan, draw request
        while (pend_r != pend_w) {
            __syncwarp();
            const int b = S.pend[pend_r % PEND];
            const float T = __ldg(P.temperature + b);
            int jb = -1;
            if (temperature_valid(T) && T > 0.0f) {
                for (int q = 0; q < NJ; ++q)
                    if (jb < 0 && vld(S.jobs[q].state) == 0)
                        jb = q;
                if (jb < 0)
                    break;  // every job slot busy: retry after a draw finishes
            }
            __threadfence();  // the sequence's partials come from other CTAs
            sequence_scan<DT>(P, S, b, jb, lane);
            ++pend_r;
            progress = true;
        }
        int busy = 0;
        for (int q = 0; q < NJ; ++q)
            busy += (vld(S.jobs[q].state) != 0) ? 1 : 0;
        if (lane == 0)
            vst(S.backlog, (pend_w - pend_r) + busy);
        // 4. done when the producer has issued its last stats tile and all of
        //    them, and every sequence this CTA owns, are finished
        if (vld(S.drain) && S.ev_r == vld(S.stats_issued) && pend_r == pend_w && busy == 0) {
            if (lane == 0)
                vst(S.finish, 1);
            break;
        }
        if (progress) {
            last_progress = globaltimer();
        } else if (globaltimer() - last_progress > WAIT_NS) {
            if (lane == 0)
                raise_abort(S, hdr);
            break;
        } else {
            __nanosleep(32);
        }
    }
    __syncwarp();
    // the last CTA to finish re-arms the tile counter for the next call
    if (lane == 0) {
        __threadfence();
        const unsigned int done = atomicAdd(&hdr->ctas_done, 1u);
        if (done == gridDim.x - 1) {
            atomicExch(&hdr->tile_counter, 0u);
            atomicExch(&hdr->ctas_done, 0u);
        }
    }
}

// ------------------------------------------------------------------ host side

struct DevCache {
    int sms = 0;
    int ctas_per_sm[2] = {0, 0};
    bool attr_set[2] = {false, false};
};
DevCache g_dev[64];

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool sizes_ok(int32_t B, int32_t k, int32_t V, int32_t dtype)
{
    return B >= 0 && k >= 1 && k <= SPEC_MAX_K && V >= 2 && V <= SPEC_MAX_V &&
           (dtype == SPEC_F32 || dtype == SPEC_BF16);
}

int tile_elems(int32_t dtype) { return TILE_BYTES / (dtype == SPEC_F32 ? 4 : 2); }

struct WsLayout {
    size_t counters, partials, chunks, chunk_stride, total, NS, DS;
};

// header | per-sequence tickets | one 16-byte partial per stats tile |
// per-sequence inverse-CDF chunk totals
WsLayout ws_layout(int32_t B, int32_t k, int32_t V, int32_t dtype)
{
    WsLayout w;
    const size_t te = tile_elems(dtype);
    w.NS = ((size_t)V + te - 1) / te;
    w.DS = ((size_t)V + te / 2 - 1) / (te / 2);
    const size_t tiles = (size_t)B * (2 * (size_t)k + 1) * w.NS;
    w.counters = 256;
    w.partials = w.counters + align_up((size_t)B * 4, 256);
    w.chunks = align_up(w.partials + tiles * 16, 256);
    w.chunk_stride = align_up(w.DS * UD * NCW, 32);  // floats, 128-byte rows
    w.total = w.chunks + (size_t)B * w.chunk_stride * 4;
    return w;
}

size_t ws_bytes(int32_t B, int32_t k, int32_t V, int32_t dtype)
{
    return ws_layout(B, k, V, dtype).total;
}

int launch(const void *target, const void *draft, const int32_t *tokens, const float *ua,
           const float *ur, const float *temp, int32_t *out_tokens, int32_t *out_n,
           float *out_probs, int32_t B, int32_t k, int32_t V, int32_t dtype, void *ws,
           size_t ws_size, void *stream)
{
    if (!sizes_ok(B, k, V, dtype))
        return SPEC_EINVAL;
    if (B == 0)
        return SPEC_OK;
    if (!target || !draft || !tokens || !ua || !ur || !temp || !out_tokens || !out_n || !ws)
        return SPEC_EINVAL;
    if ((reinterpret_cast<uintptr_t>(target) & 15) || (reinterpret_cast<uintptr_t>(draft) & 15) ||
        (reinterpret_cast<uintptr_t>(ws) & 15) || (reinterpret_cast<uintptr_t>(tokens) & 3) ||
        (reinterpret_cast<uintptr_t>(ua) & 3) || (reinterpret_cast<uintptr_t>(ur) & 3) ||
        (reinterpret_cast<uintptr_t>(temp) & 3) || (reinterpret_cast<uintptr_t>(out_tokens) & 3) ||
        (reinterpret_cast<uintptr_t>(out_n) & 3) || (reinterpret_cast<uintptr_t>(out_probs) & 3))
        return SPEC_EINVAL;
    const WsLayout lay = ws_layout(B, k, V, dtype);
    if (ws_size < lay.total)
        return SPEC_ENOSPACE;
    const size_t NS = lay.NS;
    const size_t total = (size_t)B * (2 * (size_t)k + 1) * NS;
    if (total >= 0x7fffffffull)
        return SPEC_EINVAL;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SPEC_ECUDA;
    DevCache &dc = g_dev[dev];
    const int di = (dtype == SPEC_F32) ? 0 : 1;
    const void *fn = (dtype == SPEC_F32) ? (const void *)spec_verify_kernel<SPEC_F32>
                                         : (const void *)spec_verify_kernel<SPEC_BF16>;
    if (!dc.attr_set[di]) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_BYTES) != cudaSuccess)
            return SPEC_ECUDA;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, NTHREADS, SMEM_BYTES) != cudaSuccess)
            return SPEC_ECUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SPEC_ECUDA;
        dc.sms = sms;
        dc.ctas_per_sm[di] = n > 0 ? n : 1;
        dc.attr_set[di] = true;
    }
    const size_t resident = (size_t)dc.sms * dc.ctas_per_sm[di];
    const unsigned int grid = (unsigned int)(total < resident ? total : resident);

    Params P;
    P.target = target;
    P.draft = draft;
    P.tokens = tokens;
    P.u_accept = ua;
    P.u_resample = ur;
    P.temperature = temp;
    P.out_tokens = out_tokens;
    P.out_num_accepted = out_n;
    P.out_probs = out_probs;
    P.ws = reinterpret_cast<uint8_t *>(ws);
    P.seq_count = reinterpret_cast<unsigned int *>(P.ws + lay.counters);
    P.part = reinterpret_cast<float4 *>(P.ws + lay.partials);
    P.chunks = reinterpret_cast<float *>(P.ws + lay.chunks);
    P.B = B;
    P.k = k;
    P.V = V;
    P.NS = (int)NS;
    P.rows = 2 * k + 1;
    P.DS = (int)lay.DS;
    P.chunk_stride = (int)lay.chunk_stride;
    P.total_tiles = (unsigned int)total;
    const size_t es = (dtype == SPEC_F32) ? 4 : 2;
    P.target_bytes = (unsigned long long)B * (k + 1) * (unsigned long long)V * es;
    P.draft_bytes = (unsigned long long)B * k * (unsigned long long)V * es;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == SPEC_F32)
        spec_verify_kernel<SPEC_F32><<<grid, NTHREADS, SMEM_BYTES, st>>>(P);
    else
        spec_verify_kernel<SPEC_BF16><<<grid, NTHREADS, SMEM_BYTES, st>>>(P);
    if (cudaPeekAtLastError() != cudaSuccess) {
        (void)cudaGetLastError();
        return SPEC_ECUDA;
    }
    return SPEC_OK;
}

}  // namespace

static_assert(SPEC_MAX_V / (NT * 4) + UD <= MAXBLK, "CDF blocks must cover the largest vocabulary");

// ---------------------------------------------------------------- C ABI

extern "C" {

int32_t spec_verify_abi_version(void) { return SPEC_VERIFY_ABI_VERSION; }

const char *spec_verify_strerror(int32_t status)
{
    switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_EINVAL: return "invalid argument (null pointer, size out of range, misalignment or dtype)";
    case SPEC_ECUDA: return "CUDA runtime error or launch failure";
    case SPEC_ENOSPACE: return "workspace or arena too small";
    default: return "unknown status";
    }
}

size_t spec_verify_workspace_size(int32_t B, int32_t k, int32_t V, int32_t dtype)
{
    if (!sizes_ok(B, k, V, dtype))
        return 0;
    return ws_bytes(B, k, V, dtype);
}

int32_t spec_verify_workspace_reset(void *workspace, size_t workspace_bytes, void *stream)
{
    if (!workspace)
        return SPEC_EINVAL;
    if (cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SPEC_ECUDA;
    return SPEC_OK;
}

int32_t spec_verify(const void *target_logits, const void *draft_logits,
                    const int32_t *draft_tokens, const float *u_accept,
                    const float *u_resample, const float *temperature,
                    int32_t *out_tokens, int32_t *out_num_accepted,
                    int32_t B, int32_t k, int32_t V, int32_t dtype,
                    void *workspace, size_t workspace_bytes, void *stream)
{
    return launch(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature,
                  out_tokens, out_num_accepted, nullptr, B, k, V, dtype, workspace,
                  workspace_bytes, stream);
}

int32_t spec_verify_probs(const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *u_accept,
                          const float *u_resample, const float *temperature,
                          int32_t *out_tokens, int32_t *out_num_accepted, float *out_probs,
                          int32_t B, int32_t k, int32_t V, int32_t dtype,
                          void *workspace, size_t workspace_bytes, void *stream)
{
    if (!out_probs && B > 0)
        return SPEC_EINVAL;
    return launch(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature,
                  out_tokens, out_num_accepted, out_probs, B, k, V, dtype, workspace,
                  workspace_bytes, stream);
}

int32_t spec_verify_read_status(const void *workspace, int32_t *status, void *stream)
{
    if (!workspace || !status)
        return SPEC_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const WsHeader *hdr = reinterpret_cast<const WsHeader *>(workspace);
    if (cudaMemcpyAsync(status, &hdr->status, sizeof(int32_t), cudaMemcpyDeviceToHost, st) !=
        cudaSuccess)
        return SPEC_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return SPEC_ECUDA;
    return SPEC_OK;
}

size_t spec_verify_host_arena_size(int32_t B, int32_t k, int32_t V, int32_t dtype)
{
    if (!sizes_ok(B, k, V, dtype))
        return 0;
    const size_t es = (dtype == SPEC_F32) ? 4 : 2;
    size_t n = 0;
    n += align_up((size_t)B * (k + 1) * V * es, 256);  // target
    n += align_up((size_t)B * k * V * es, 256);        // draft
    n += align_up((size_t)B * k * 4, 256);             // tokens
    n += align_up((size_t)B * k * 4, 256);             // u_accept
    n += align_up((size_t)B * 4, 256);                 // u_resample
    n += align_up((size_t)B * 4, 256);                 // temperature
    n += align_up((size_t)B * (k + 1) * 4, 256);       // out_tokens
    n += align_up((size_t)B * 4, 256);                 // out_num_accepted
    n += align_up(ws_bytes(B, k, V, dtype), 256);      // workspace
    return n;
}

int32_t spec_verify_host(const void *target_logits, const void *draft_logits,
                         const int32_t *draft_tokens, const float *u_accept,
                         const float *u_resample, const float *temperature,
                         int32_t *out_tokens, int32_t *out_num_accepted,
                         int32_t B, int32_t k, int32_t V, int32_t dtype,
                         void *device_arena, size_t arena_bytes, void *stream)
{
    if (!sizes_ok(B, k, V, dtype))
        return SPEC_EINVAL;
    if (B == 0)
        return SPEC_OK;
    if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_resample ||
        !temperature || !out_tokens || !out_num_accepted || !device_arena)
        return SPEC_EINVAL;
    if (reinterpret_cast<uintptr_t>(device_arena) & 255)
        return SPEC_EINVAL;
    if (arena_bytes < spec_verify_host_arena_size(B, k, V, dtype))
        return SPEC_ENOSPACE;
    const size_t es = (dtype == SPEC_F32) ? 4 : 2;
    uint8_t *a = reinterpret_cast<uint8_t *>(device_arena);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = a + off;
        off += align_up(bytes, 256);
        return p;
    };
    const size_t bt = (size_t)B * (k + 1) * V * es, bd = (size_t)B * k * V * es;
    uint8_t *d_t = take(bt), *d_d = take(bd);
    uint8_t *d_g = take((size_t)B * k * 4), *d_ua = take((size_t)B * k * 4);
    uint8_t *d_ur = take((size_t)B * 4), *d_T = take((size_t)B * 4);
    uint8_t *d_ot = take((size_t)B * (k + 1) * 4), *d_on = take((size_t)B * 4);
    const size_t wsb = ws_bytes(B, k, V, dtype);
    uint8_t *d_ws = take(wsb);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const struct {
        void *dst;
        const void *src;
        size_t n;
    } cps[] = {{d_t, target_logits, bt},       {d_d, draft_logits, bd},
               {d_g, draft_tokens, (size_t)B * k * 4}, {d_ua, u_accept, (size_t)B * k * 4},
               {d_ur, u_resample, (size_t)B * 4},    {d_T, temperature, (size_t)B * 4}};
    for (const auto &c : cps)
        if (cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return SPEC_ECUDA;
    if (cudaMemsetAsync(d_ws, 0, wsb, st) != cudaSuccess)
        return SPEC_ECUDA;
    int rc = launch(d_t, d_d, reinterpret_cast<const int32_t *>(d_g),
                    reinterpret_cast<const float *>(d_ua), reinterpret_cast<const float *>(d_ur),
                    reinterpret_cast<const float *>(d_T), reinterpret_cast<int32_t *>(d_ot),
                    reinterpret_cast<int32_t *>(d_on), nullptr, B, k, V, dtype, d_ws, wsb, stream);
    if (rc != SPEC_OK)
        return rc;
    if (cudaMemcpyAsync(out_tokens, d_ot, (size_t)B * (k + 1) * 4, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaMemcpyAsync(out_num_accepted, d_on, (size_t)B * 4, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess)
        return SPEC_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return SPEC_ECUDA;
    return SPEC_OK;
}

}  // extern "C"
