// spec_verify.cu -- GB300 (sm_103a) kernels and C ABI for batched
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
// Design (one persistent kernel per call):
//   * Work unit = tile: one 32 KB segment of one logits row (row = a target or
//     draft position of one sequence).  Tiles are numbered sequence-major and
//     handed out by a global atomic counter, so every CTA streams a fair share
//     and the tiles of one sequence are read close together in time.
//   * Each CTA = 1 producer warp + 8 consumer warps.  The producer's elected
//     lane claims tiles and moves them with cp.async.bulk (the TMA bulk-copy
//     path) into a 3-stage shared-memory ring guarded by mbarriers.  Two CTAs
//     fit per SM, so up to 6 tiles (192 KB) per SM are in flight.
//   * Consumers compute, per tile, the row statistics of the temperature
//     softmax: maximum m, lowest-index argmax and Z = sum 2^((x-m)*log2(e)/T)
//     (one exp per element, max taken over the thread's registers first), and
//     write a 16-byte partial to the workspace.
//   * A per-sequence ticket (atomic counter) elects the CTA that finishes a
//     sequence's last tile.  That CTA combines the partials, runs the accept
//     scan (first rejection) and draws the correction / bonus token by
//     inverse CDF over the rows it needs, which are still resident in L2.
//   * Reduction orders depend only on row-relative indices, never on which
//     CTA handled a tile or on the row's address, so bit-identical target and
//     draft rows give bit-identical statistics (their ratio is exactly 1).
//   * Every wait is bounded: a timed-out wait records SPEC_DEV_WAIT_TIMEOUT in
//     the workspace and the kernel returns; nothing traps.
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "spec_verify.h"

namespace {

constexpr int NCW = 8;                          // consumer warps
constexpr int NT = NCW * 32;                    // consumer threads
constexpr int NTHREADS = NT + 32;               // + one producer warp
constexpr int STAGES = 3;                       // shared-memory ring depth
constexpr int TILE_BYTES = 32768;               // one tile of one row
constexpr int SLOT_BYTES = TILE_BYTES + 128;    // room for a misaligned head/tail
constexpr int U = TILE_BYTES / (NT * 16);       // 16-byte vectors per consumer per tile
constexpr int MAX_ROWS = 2 * SPEC_MAX_K + 1;
constexpr int MAXB = 1024;                      // draw blocks (one vector per thread each)
constexpr int DRAW_G = 2;                       // draw blocks loaded per step
constexpr float LOG2E = 1.4426950408889634f;
constexpr int BAR_CONSUMERS = 1;                // named barrier id for consumer warps
constexpr unsigned long long WAIT_NS = 2000000000ull;  // 2 s bound on any wait

static_assert(U * NT * 16 == TILE_BYTES, "tile must split evenly over consumers");

struct WsHeader {
    unsigned int tile_counter;
    unsigned int ctas_done;
    int status;
    unsigned int pad[61];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct TileInfo {
    int tile;     // -1 = no more tiles
    int b;        // sequence
    int rsq;      // row in sequence: 0..k target, k+1..2k draft
    int seg;      // segment within the row
    int mode;     // 0 skip (not read), 1 greedy (max/argmax), 2 sampling (max/argmax/Z)
    float c;      // log2(e) / T
    int phase;    // bytes from the copy start to the tile's first element
    int ncopied;  // bytes present in the slot
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
    int B, k, V;
    int NS;            // tiles per row
    int rows;          // rows per sequence (2k+1)
    int nb;            // draw blocks per row
    unsigned int total_tiles;
    unsigned long long target_bytes, draft_bytes;
};

struct Tail {
    float rm[MAX_ROWS];
    float rZ[MAX_ROWS];
    int rarg[MAX_ROWS];
    int rbad[MAX_ROWS];
    float btot[MAXB];
    float wt[2][DRAW_G][NCW];
    int cand[NCW];
    int lastpos[NCW];
    int j, err, token, bstar, mode;
    float base, uR, R;
};

struct Smem {
    unsigned long long full[STAGES];
    unsigned long long empty[STAGES];
    TileInfo info[STAGES];
    float4 red[NCW];
    int flag;
    int pad[3];
    Tail tail;
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

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync %0, %1;" ::"n"(BAR_CONSUMERS), "n"(NT) : "memory");
}

// Consumer barrier that also ORs a predicate over the consumer threads.
__device__ __forceinline__ bool consumers_sync_or(bool pred)
{
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)pred), "n"(BAR_CONSUMERS), "n"(NT)
        : "memory");
    return out != 0;
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

// ----------------------------------------------------------- tile statistics

// Load the raw 16-byte vector `v` (row-relative vector index) of a tile from
// its shared-memory slot, or element by element when the slot's data is not
// 16-byte aligned with the row, or lies past the bytes that were copied.
template <int DT>
__device__ __forceinline__ uint4 tile_vec(const Params &P, const TileInfo &ti,
                                          const uint8_t *slot, int v, int e0, int e1,
                                          bool fast)
{
    using L = Lg<DT>;
    if (fast)
        return ld_shared_v4(slot + (size_t)(v * L::VEC - e0) * L::ES);
    uint4 r = neg_inf_vec(L::NEG_INF_WORD);
    const bool is_target = ti.rsq <= P.k;
    const void *arr = is_target ? P.target : P.draft;
    const size_t row = is_target ? (size_t)ti.b * (P.k + 1) + ti.rsq
                                 : (size_t)ti.b * P.k + (ti.rsq - P.k - 1);
#pragma unroll
    for (int j = 0; j < L::VEC; ++j) {
        const int e = v * L::VEC + j;
        if (e >= e0 && e < e1) {
            const int off = ti.phase + (e - e0) * L::ES;
            uint32_t bits;
            if (off + L::ES <= ti.ncopied)
                bits = L::bits_at(slot + off);
            else
                bits = __float_as_uint(L::load1(arr, row * (size_t)P.V + e)) >> (DT == SPEC_BF16 ? 16 : 0);
            L::put(r, j, bits);
        }
    }
    return r;
}

// Per-thread statistics of one tile: the thread owns vectors tid, tid+NT, ...
template <int DT>
__device__ __forceinline__ void tile_thread_stats(const Params &P, const TileInfo &ti,
                                                  const uint8_t *slot, int tid, float &m_out,
                                                  float &s_out, int &idx_out)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    constexpr int SEG = TILE_BYTES / L::ES;
    const int e0 = ti.seg * SEG;
    const int e1 = min(P.V, e0 + SEG);
    const int v0 = e0 / VEC;
    const int v1 = (e1 + VEC - 1) / VEC;
    const int nbytes = (e1 - e0) * L::ES;
    const bool fast = (ti.phase == 0) && ((nbytes & 15) == 0) && (ti.ncopied >= nbytes);

    uint4 raw[U];
    float vmax[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int v = v0 + tid + u * NT;
        if (v < v1) {
            raw[u] = tile_vec<DT>(P, ti, slot, v, e0, e1, fast);
        } else {
            raw[u] = neg_inf_vec(L::NEG_INF_WORD);
        }
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

    // lowest row-relative index attaining m (INT_MAX if this thread has no data)
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
    if (ti.mode == 2 && m != -INFINITY) {
        const float c = ti.c;
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

// ------------------------------------------------------------------ the draw

// w(e) for one vector: residual max(0, p - q) (mode 1) or unnormalised p (mode 2)
struct DrawRow {
    const void *rowT;
    const void *rowD;
    bool alignedT, alignedD;
    float mt, rzt, md, rzd, c;
    int mode;
};

template <int DT>
__device__ __forceinline__ uint4 row_vec(const void *row, bool aligned, int v, int V)
{
    using L = Lg<DT>;
    const int e = v * L::VEC;
    if (aligned && e + L::VEC <= V)
        return __ldg(reinterpret_cast<const uint4 *>(row) + v);
    uint4 r = neg_inf_vec(L::NEG_INF_WORD);
#pragma unroll
    for (int j = 0; j < L::VEC; ++j)
        if (e + j < V)
            L::put(r, j, __float_as_uint(L::load1(row, (size_t)(e + j))) >> (DT == SPEC_BF16 ? 16 : 0));
    return r;
}

template <int DT>
__device__ __forceinline__ void draw_weights(const DrawRow &D, const uint4 &rt, const uint4 &rd,
                                             float (&w)[Lg<DT>::VEC])
{
    using L = Lg<DT>;
    float xt[L::VEC];
    L::unpack(rt, xt);
    if (D.mode == 1) {
        float xd[L::VEC];
        L::unpack(rd, xd);
#pragma unroll
        for (int j = 0; j < L::VEC; ++j) {
            const float p = ex2((xt[j] - D.mt) * D.c) * D.rzt;
            const float q = ex2((xd[j] - D.md) * D.c) * D.rzd;
            w[j] = fmaxf(p - q, 0.0f);
        }
    } else {
#pragma unroll
        for (int j = 0; j < L::VEC; ++j)
            w[j] = ex2((xt[j] - D.mt) * D.c);
    }
}

// Thread-level inclusive sums of one vector's weights, then the warp-level
// inclusive scan of thread totals (Kogge-Stone) and its exclusive shift.
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

// Inverse-CDF draw over one row (or a residual row pair) by all consumer
// threads.  C(x) is a fixed hierarchical prefix sum (thread, warp, block,
// then blocks left to right); R is its own final value; the token is the
// smallest x with w(x) > 0 and C(x) > u * R.
template <int DT>
__device__ int draw_token(const Params &P, const DrawRow &D, float u, Tail &tl, int tid,
                          bool &zero_mass)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    const int lane = tid & 31, warp = tid >> 5;
    const int nb = P.nb;

    // pass A: block totals, DRAW_G blocks per step
    for (int g0 = 0, gp = 0; g0 < nb; g0 += DRAW_G, gp ^= 1) {
        uint4 rt[DRAW_G], rd[DRAW_G];
#pragma unroll
        for (int g = 0; g < DRAW_G; ++g) {
            const int v = (g0 + g) * NT + tid;
            if (g0 + g < nb) {
                rt[g] = row_vec<DT>(D.rowT, D.alignedT, v, P.V);
                rd[g] = (D.mode == 1) ? row_vec<DT>(D.rowD, D.alignedD, v, P.V) : rt[g];
            }
        }
        float tau[DRAW_G], excl[DRAW_G];
#pragma unroll
        for (int g = 0; g < DRAW_G; ++g) {
            tau[g] = 0.0f;
            excl[g] = 0.0f;
            if (g0 + g < nb) {
                float w[VEC];
                draw_weights<DT>(D, rt[g], rd[g], w);
                float s = 0.0f;
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    s = s + w[j];
                tau[g] = s;
                float incl;
                warp_scan(s, lane, incl, excl[g]);
                if (lane == 31)
                    tl.wt[gp][g][warp] = incl;
            }
        }
        consumers_sync();
        if (tid == NT - 1) {
#pragma unroll
            for (int g = 0; g < DRAW_G; ++g) {
                if (g0 + g < nb) {
                    float om = 0.0f;
                    for (int w2 = 0; w2 < NCW - 1; ++w2)
                        om = om + tl.wt[gp][g][w2];
                    tl.btot[g0 + g] = (om + excl[g]) + tau[g];
                }
            }
        }
    }
    consumers_sync();

    // R and the block holding the crossing, by one thread, left to right
    if (tid == 0) {
        float base = 0.0f;
        for (int bk = 0; bk < nb; ++bk)
            base = base + tl.btot[bk];
        const float R = base;
        const float uR = u * R;
        int bstar = nb - 1;
        float bb = 0.0f;
        base = 0.0f;
        for (int bk = 0; bk < nb; ++bk) {
            const float nxt = base + tl.btot[bk];
            if (nxt > uR) {
                bstar = bk;
                bb = base;
                break;
            }
            base = nxt;
        }
        tl.R = R;
        tl.uR = uR;
        tl.bstar = bstar;
        tl.base = bb;
    }
    consumers_sync();
    if (!(tl.R > 0.0f)) {
        zero_mass = true;
        return -1;
    }
    zero_mass = false;

    // pass B: the chosen block, element by element
    const int bstar = tl.bstar;
    const int v = bstar * NT + tid;
    const uint4 rt = row_vec<DT>(D.rowT, D.alignedT, v, P.V);
    const uint4 rd = (D.mode == 1) ? row_vec<DT>(D.rowD, D.alignedD, v, P.V) : rt;
    float w[VEC];
    draw_weights<DT>(D, rt, rd, w);
    float sacc[VEC];
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        s = s + w[j];
        sacc[j] = s;
    }
    float incl, excl;
    warp_scan(s, lane, incl, excl);
    if (lane == 31)
        tl.wt[0][0][warp] = incl;
    consumers_sync();
    float om = 0.0f;
    for (int w2 = 0; w2 < warp; ++w2)
        om = om + tl.wt[0][0][w2];
    const float pre = om + excl;
    const float base = tl.base, uR = tl.uR;
    int cand = INT_MAX, lastp = -1;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        const int e = v * VEC + j;
        if (w[j] > 0.0f) {
            lastp = e;
            const float C = base + (pre + sacc[j]);
            if (cand == INT_MAX && C > uR)
                cand = e;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
        lastp = max(lastp, __shfl_xor_sync(0xffffffffu, lastp, o));
    }
    if (lane == 0) {
        tl.cand[warp] = cand;
        tl.lastpos[warp] = lastp;
    }
    consumers_sync();
    int c2 = INT_MAX, l2 = -1;
    for (int w2 = 0; w2 < NCW; ++w2) {
        c2 = min(c2, tl.cand[w2]);
        l2 = max(l2, tl.lastpos[w2]);
    }
    consumers_sync();  // tl.* reused by the caller
    return (c2 != INT_MAX) ? c2 : l2;
}

// ------------------------------------------------------------ sequence tail

__device__ __forceinline__ bool temperature_valid(float T)
{
    return !(isnan(T) || T < 0.0f || isinf(T) || (T > 0.0f && T < FLT_MIN));
}

template <int DT>
__device__ __forceinline__ void sequence_tail(const Params &P, int b, Tail &tl, int tid)
{
    using L = Lg<DT>;
    const int lane = tid & 31, warp = tid >> 5;
    const int k = P.k, V = P.V;
    const float T = __ldg(P.temperature + b);
    const bool tvalid = temperature_valid(T);
    const bool greedy = tvalid && T == 0.0f;
    const float c = (tvalid && !greedy) ? LOG2E / T : 0.0f;
    const float4 *part = reinterpret_cast<const float4 *>(P.ws + 256 + (((size_t)P.B * 4 + 255) & ~(size_t)255));

    // 1. combine tile partials into row statistics
    const int nrows = tvalid ? (greedy ? k + 1 : P.rows) : 0;
    for (int r = warp; r < nrows; r += NCW) {
        float m = -INFINITY, s = 0.0f;
        int idx = INT_MAX;
        for (int sg = lane; sg < P.NS; sg += 32) {
            const float4 pv = __ldcg(part + ((size_t)b * P.rows + r) * P.NS + sg);
            const float pm = pv.x, ps = pv.y;
            const int pi = __float_as_int(pv.z);
            const float mn = fmax_nan(m, pm);
            if (!greedy)
                s = rescale(s, m, mn, c) + rescale(ps, pm, mn, c);
            idx = (m == mn && pm == mn) ? min(idx, pi) : (pm == mn ? pi : idx);
            m = mn;
        }
        warp_combine(m, s, idx, c, !greedy);
        if (lane == 0) {
            tl.rm[r] = m;
            tl.rZ[r] = s;
            tl.rarg[r] = idx;
            tl.rbad[r] = (isnan(m) || isinf(m)) ? 1 : 0;  // NaN, +inf, or all -inf
        }
    }
    consumers_sync();

    // 2. accept scan (warp 0; lane i tests position i)
    if (warp == 0) {
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
                if (tl.rbad[r])
                    err = true;
            err = __any_sync(0xffffffffu, err);
        }
        int j = k, token = -1;
        if (!err) {
            if (greedy) {
                fail = (lane < k) && (g != tl.rarg[lane]);
            } else if (lane < k) {
                const size_t rt = (size_t)b * (k + 1) + lane, rd = (size_t)b * k + lane;
                const float lt = L::load1(P.target, rt * V + g);
                const float ld = L::load1(P.draft, rd * V + g);
                const float mt = tl.rm[lane], zt = tl.rZ[lane];
                const float md = tl.rm[k + 1 + lane], zd = tl.rZ[k + 1 + lane];
                qzero = (ld == -INFINITY);
                const float dt = lt - mt, dd = ld - md;
                const float x = (dt - dd) * c;
                const float ratio = ((x == 0.0f) ? 1.0f : ex2(x)) * (zd / zt);
                const float ua = __ldg(P.u_accept + (size_t)b * k + lane);
                const bool accept = (ratio >= 1.0f) || (ua < ratio);
                fail = qzero || !accept;
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
                token = tl.rarg[j];
            }
        }
        if (P.out_probs && (err || greedy) && lane < k) {
            P.out_probs[((size_t)b * k + lane) * 2 + 0] = __int_as_float(0x7fc00000);
            P.out_probs[((size_t)b * k + lane) * 2 + 1] = __int_as_float(0x7fc00000);
        }
        if (lane == 0) {
            tl.err = err ? 1 : 0;
            tl.j = j;
            tl.token = token;
        }
    }
    consumers_sync();

    // 3. the draw (sampling mode)
    const int err = tl.err;
    const int j = tl.j;
    if (!err && !greedy) {
        DrawRow D;
        D.c = c;
        const size_t rt = (size_t)b * (k + 1) + j;
        D.rowT = reinterpret_cast<const uint8_t *>(P.target) + rt * (size_t)V * L::ES;
        D.alignedT = ((reinterpret_cast<uintptr_t>(D.rowT) & 15) == 0);
        D.mt = tl.rm[j];
        D.rzt = 1.0f / tl.rZ[j];
        if (j < k) {
            const size_t rd = (size_t)b * k + j;
            D.rowD = reinterpret_cast<const uint8_t *>(P.draft) + rd * (size_t)V * L::ES;
            D.alignedD = ((reinterpret_cast<uintptr_t>(D.rowD) & 15) == 0);
            D.md = tl.rm[k + 1 + j];
            D.rzd = 1.0f / tl.rZ[k + 1 + j];
            D.mode = 1;
        } else {
            D.rowD = D.rowT;
            D.alignedD = D.alignedT;
            D.md = D.mt;
            D.rzd = D.rzt;
            D.mode = 2;
        }
        const float u = __ldg(P.u_resample + b);
        bool zero_mass = false;
        int tok = draw_token<DT>(P, D, u, tl, tid, zero_mass);
        if (zero_mass && D.mode == 1) {
            // rounding-only: the residual vanished; sample p_j instead
            D.mode = 2;
            tok = draw_token<DT>(P, D, u, tl, tid, zero_mass);
        }
        if (tid == 0) {
            if (zero_mass || tok < 0)
                tl.err = 1;
            tl.token = tok;
        }
        consumers_sync();
    }

    // 4. outputs
    if (warp == 0) {
        const int e2 = tl.err;
        const int tok = tl.token;
        for (int i = lane; i <= k; i += 32) {
            int o;
            if (e2)
                o = -1;
            else if (i < j)
                o = __ldg(P.tokens + (size_t)b * k + i);
            else if (i == j)
                o = tok;
            else
                o = -1;
            P.out_tokens[(size_t)b * (k + 1) + i] = o;
        }
        if (lane == 0) {
            P.out_num_accepted[b] = e2 ? -1 : j;
            unsigned int *seq_count = reinterpret_cast<unsigned int *>(P.ws + 256);
            atomicExch(seq_count + b, 0u);  // ready for the next call
        }
    }
    consumers_sync();
}

// ------------------------------------------------------------------- kernel

template <int DT>
__global__ void __launch_bounds__(NTHREADS, 2) spec_verify_kernel(const Params P)
{
    using L = Lg<DT>;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *slots = smem_raw;
    Smem &S = *reinterpret_cast<Smem *>(smem_raw + (size_t)STAGES * SLOT_BYTES);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(P.ws);
    unsigned int *seq_count = reinterpret_cast<unsigned int *>(P.ws + 256);
    float4 *part = reinterpret_cast<float4 *>(P.ws + 256 + (((size_t)P.B * 4 + 255) & ~(size_t)255));

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], NCW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    constexpr int SEG = TILE_BYTES / L::ES;
    const unsigned int tiles_per_seq = (unsigned int)P.rows * (unsigned int)P.NS;

    if (warp == NCW) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            unsigned int t = atomicAdd(&hdr->tile_counter, 1u);
            while (true) {
                if (!mbar_wait(&S.empty[stage], phase ^ 1u)) {
                    atomicExch(&hdr->status, SPEC_DEV_WAIT_TIMEOUT);
                    // let the copies already issued land before leaving
                    for (int s = 0; s < STAGES; ++s)
                        (void)mbar_wait(&S.full[s], (s < stage) ? phase : (phase ^ 1u));
                    break;
                }
                TileInfo &ti = S.info[stage];
                if (t >= P.total_tiles) {
                    ti.tile = -1;
                    mbar_arrive(&S.full[stage]);
                    break;
                }
                const int b = (int)(t / tiles_per_seq);
                const unsigned int rem = t - (unsigned int)b * tiles_per_seq;
                const int rsq = (int)(rem / (unsigned int)P.NS);
                const int seg = (int)(rem - (unsigned int)rsq * (unsigned int)P.NS);
                const float T = __ldg(P.temperature + b);
                int mode;
                if (!temperature_valid(T))
                    mode = 0;
                else if (T == 0.0f)
                    mode = (rsq <= P.k) ? 1 : 0;  // greedy never reads draft rows
                else
                    mode = 2;
                ti.tile = (int)t;
                ti.b = b;
                ti.rsq = rsq;
                ti.seg = seg;
                ti.mode = mode;
                ti.c = (mode == 2) ? LOG2E / T : 0.0f;
                uint32_t bytes = 0;
                int ph = 0;
                if (mode != 0) {
                    const bool is_target = rsq <= P.k;
                    const uint8_t *arr = reinterpret_cast<const uint8_t *>(is_target ? P.target : P.draft);
                    const unsigned long long arr_bytes = is_target ? P.target_bytes : P.draft_bytes;
                    const size_t row = is_target ? (size_t)b * (P.k + 1) + rsq
                                                 : (size_t)b * P.k + (rsq - P.k - 1);
                    const int e0 = seg * SEG;
                    const int e1 = min(P.V, e0 + SEG);
                    const unsigned long long start = ((unsigned long long)row * P.V + e0) * L::ES;
                    const unsigned long long end = ((unsigned long long)row * P.V + e1) * L::ES;
                    const unsigned long long a0 = start & ~15ull;
                    unsigned long long a1 = (end + 15) & ~15ull;
                    const unsigned long long lim = arr_bytes & ~15ull;
                    if (a1 > lim)
                        a1 = lim;
                    ph = (int)(start - a0);
                    bytes = (a1 > a0) ? (uint32_t)(a1 - a0) : 0u;
                    ti.phase = ph;
                    ti.ncopied = (int)bytes;
                    if (bytes) {
                        mbar_arrive_expect_tx(&S.full[stage], bytes);
                        bulk_copy_g2s(slots + (size_t)stage * SLOT_BYTES, arr + a0, bytes, &S.full[stage]);
                    } else {
                        mbar_arrive(&S.full[stage]);
                    }
                } else {
                    ti.phase = 0;
                    ti.ncopied = 0;
                    mbar_arrive(&S.full[stage]);
                }
                t = atomicAdd(&hdr->tile_counter, 1u);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        // ---------------------------------------------------------- consumers
        int stage = 0;
        uint32_t phase = 0;
        int tail_b = -1;  // sequence whose tail this CTA owes, run between tiles
        while (true) {
            if (tail_b >= 0) {
                sequence_tail<DT>(P, tail_b, S.tail, tid);
                tail_b = -1;
            }
            const bool ok = mbar_wait(&S.full[stage], phase);
            if (consumers_sync_or(!ok)) {
                if (tid == 0)
                    atomicExch(&hdr->status, SPEC_DEV_WAIT_TIMEOUT);
                break;
            }
            const TileInfo ti = S.info[stage];
            if (ti.tile < 0)
                break;
            float m = -INFINITY, s = 0.0f;
            int idx = INT_MAX;
            if (ti.mode != 0)
                tile_thread_stats<DT>(P, ti, slots + (size_t)stage * SLOT_BYTES, tid, m, s, idx);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&S.empty[stage]);
            if (ti.mode != 0) {
                warp_combine(m, s, idx, ti.c, ti.mode == 2);
                if (lane == 0)
                    S.red[warp] = make_float4(m, s, __int_as_float(idx), 0.0f);
            }
            consumers_sync();
            if (warp == 0) {
                if (ti.mode != 0) {
                    float m2 = -INFINITY, s2 = 0.0f;
                    int i2 = INT_MAX;
                    if (lane < NCW) {
                        const float4 r = S.red[lane];
                        m2 = r.x;
                        s2 = r.y;
                        i2 = __float_as_int(r.z);
                    }
                    warp_combine(m2, s2, i2, ti.c, ti.mode == 2);
                    if (lane == 0)
                        __stcg(part + (size_t)ti.b * P.rows * P.NS + (size_t)ti.rsq * P.NS + ti.seg,
                               make_float4(m2, s2, __int_as_float(i2), 0.0f));
                }
                if (lane == 0) {
                    __threadfence();
                    const unsigned int old = atomicAdd(seq_count + ti.b, 1u);
                    S.flag = (old == tiles_per_seq - 1) ? 1 : 0;
                    if (S.flag)
                        __threadfence();
                }
            }
            consumers_sync();
            if (S.flag)
                tail_b = ti.b;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // the last CTA to finish re-arms the tile counter for the next call
        if (tid == 0) {
            __threadfence();
            const unsigned int done = atomicAdd(&hdr->ctas_done, 1u);
            if (done == gridDim.x - 1) {
                atomicExch(&hdr->tile_counter, 0u);
                atomicExch(&hdr->ctas_done, 0u);
            }
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

size_t ws_bytes(int32_t B, int32_t k, int32_t V, int32_t dtype)
{
    const size_t NS = ((size_t)V + tile_elems(dtype) - 1) / tile_elems(dtype);
    const size_t tiles = (size_t)B * (2 * (size_t)k + 1) * NS;
    return 256 + align_up((size_t)B * 4, 256) + tiles * 16;
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
    const size_t need = ws_bytes(B, k, V, dtype);
    if (ws_size < need)
        return SPEC_ENOSPACE;
    const size_t NS = ((size_t)V + tile_elems(dtype) - 1) / tile_elems(dtype);
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
    P.B = B;
    P.k = k;
    P.V = V;
    P.NS = (int)NS;
    P.rows = 2 * k + 1;
    const int vec = (dtype == SPEC_F32) ? 4 : 8;
    P.nb = (int)(((size_t)V + (size_t)NT * vec - 1) / ((size_t)NT * vec));
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

static_assert(SPEC_MAX_V <= MAXB * NT * 4, "draw blocks must cover the largest vocabulary");

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
