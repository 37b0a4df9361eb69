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
// One call runs four kernels on the caller's stream; none waits on another
// CTA, so nothing in a call can deadlock:
//   1. row statistics (the HBM-bound bulk of the work): a persistent,
//      warp-specialised kernel.  A producer warp streams 32 KB row tiles with
//      cp.async.bulk (the TMA bulk-copy engine) into a 3-stage shared-memory
//      ring guarded by mbarriers; 8 consumer warps reduce them.  Four
//      consecutive tiles of a row form a super-tile: every lane accumulates
//      over it (online max / sum of exponentials), and one 16-byte partial
//      per super-tile (maximum, sum of 2^((x-m)*log2(e)/T), lowest-index
//      argmax) goes to the workspace.
//   2. accept scan: one warp per sequence folds its rows' partials, runs the
//      left-to-right accept test up to the first rejection, writes greedy and
//      error sequences' outputs and a draw job for the others.
//   3. draw tiles: the one or two rows each draw needs (the residual at the
//      rejected position, or the bonus row) are read once more; every warp
//      writes the inverse-CDF totals of its 32-lane chunks.
//   4. final search: one warp per drawing sequence walks block, chunk and
//      element running sums to the drawn token and writes the outputs.
// Reduction orders depend only on row-relative indices, never on which CTA
// or warp handled a tile or on the row's address, so bit-identical target and
// draft rows give bit-identical statistics (their ratio is exactly 1).  The
// one wait on another warp (the mbarrier ring) is bounded: a timed-out wait
// records SPEC_DEV_WAIT_TIMEOUT in the workspace and the kernel returns.
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "spec_verify.h"
#include "device_common.cuh"
#include "resolve.cuh"
#include "internal.h"

namespace {

using namespace spec_dev;

constexpr int NCW = 8;                           // consumer warps
constexpr int NT = NCW * 32;                     // consumer threads
constexpr int WARP_P = NCW;                      // producer warp
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int STAGES = 3;                        // shared-memory ring depth
constexpr int TILE_BYTES = 32768;                // one tile of one row
constexpr int SUPER = 4;                         // tiles per super-tile (one partial)
constexpr int SLOT_BYTES = TILE_BYTES + 128;     // room for a misaligned head/tail
constexpr int U = TILE_BYTES / (NT * 16);        // 16-byte vectors per consumer per tile
constexpr int HALF_BYTES = TILE_BYTES / 2;       // one row's share of a draw tile
constexpr int UD = HALF_BYTES / (NT * 16);       // inverse-CDF blocks per draw tile
constexpr int MAX_ROWS = 2 * SPEC_MAX_K + 1;
constexpr int MAXBLK = SPEC_MAX_V / (NT * 4) + UD;  // inverse-CDF blocks per row, worst case
constexpr int SCAN_WARPS = 8;                    // sequences per CTA in kernels 2 and 4

static_assert(U * NT * 16 == TILE_BYTES, "stats tile must split evenly over consumers");
static_assert(UD * NT * 16 == HALF_BYTES, "draw tile must split evenly over consumers");
static_assert(NCW * CHUNK_BYTES == TILE_BYTES, "a stats tile is one 4 KB chunk per consumer warp");
static_assert(CHUNK_UV == U, "a consumer lane holds one chunk's vectors");


enum { KIND_END = 0, KIND_STATS = 1 };
enum { MODE_SKIP = 0, MODE_GREEDY = 1, MODE_SAMPLE = 2 };   // stats work
enum { DRAW_NONE = 0, DRAW_RESIDUAL = 1, DRAW_TARGET = 2 };

// The draw of one sequence (kernel 2 -> kernels 3 and 4).  With top-k /
// top-p filtering (filt = 1), x is in the target row's kept set iff
// key(x) > kt or (key(x) == kt and x <= it), likewise for the draft row, and
// rzt / rzd are the reciprocals of the kept sets' masses.
struct alignas(16) JobRec {
    int mode, j, b, filt;
    float mt, rzt, md, rzd;
    float c, u;
    int pad0, pad1;
    long long t_row, d_row;
    unsigned int kt;
    int it;
    unsigned int kd;
    int id;
};
static_assert(sizeof(JobRec) == 80, "job record is 80 bytes");
constexpr int JOB_VECS = (int)(sizeof(JobRec) / 16);

// Top-k / top-p boundary of one row (filter kernel -> scan kernel).
struct alignas(16) FiltRec {
    unsigned int kappa;  // key of the last kept token
    int iota;            // its index (ties at kappa are kept up to it)
    float zt;            // mass of the kept set, relative to the row maximum
    int flags;           // FILT_OFF, FILT_ON, FILT_ERR
};
enum { FILT_OFF = 0, FILT_ON = 1, FILT_ERR = 2, FILT_RADIX = 3 };  // RADIX: the window
                                                                   // kernel left the row to
                                                                   // the radix search

// Order-preserving unsigned key of an fp32 bit pattern (bf16 values widen
// exactly, so their keys order the same way).
__host__ __device__ __forceinline__ unsigned int okey(unsigned int b)
{
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The key of a logit of dtype DT: for bf16 only the top 16 bits carry it (a
// widened bf16 has 16 zero low bits, which the complement of a negative
// value would turn into ones).
template <int DT>
__device__ __forceinline__ unsigned int key_of(float x)
{
    return okey(__float_as_uint(x)) & ((DT == SPEC_BF16) ? 0xffff0000u : 0xffffffffu);
}

// The logit a key was made from (a bf16 value's low 16 bits are zero).
template <int DT>
__device__ __forceinline__ float val_of_key(unsigned int key)
{
    const unsigned int b = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
    return __uint_as_float(b & ((DT == SPEC_BF16) ? 0xffff0000u : 0xffffffffu));
}

struct TileInfo {
    int kind;
    int b;         // sequence
    int rsq;       // row in sequence (0..k target, k+1..2k draft)
    int seg;       // tile of the row
    int mode;
    int last;      // last tile of its super-tile
    float c;       // log2(e) / T
    int phase0;    // bytes from the copy start to the tile's first element
    int ncopied0;  // bytes present in the slot
    int bonus;     // the bonus row of a sampling sequence: write chunk records
    int pad[2];
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
    WsHeader *hdr;
    float4 *part;      // [B][rows][NSS]
    JobRec *jobs;      // [B]
    float *chunks;     // [B][chunk_stride]
    float2 *rec;       // [B][NCH] chunk records of each sequence's bonus row
    const int32_t *top_k;  // [B] or null (filtered calls)
    const float *top_p;    // [B] or null (filtered calls)
    FiltRec *filt;     // [B][rows] (filtered calls)
    unsigned int *gkey;  // [B][rows][NS * NT] lane-group maximum keys (filtered calls
                         // with room for them; null otherwise)
    unsigned long long *kept;  // [B][rows][KF_KMAX] the kept tokens of the rows cut from
                               // group maxima, as sort keys in rank order (with gkey)
    int *kcount;               // [B][rows] their number; -1: the row was not cut there
    // exact draws of the rows whose fp32 draw is near a cell boundary
    RJob *rjob;            // [B] the listed draws (count in hdr->n_flag)
    unsigned int *rkcnt;   // [B] their counts of groups of undecided elements
    float guard_abs;       // residual draws: list when u*R is within this of a cell edge
    float guard_rel;       // bonus / target-row draws: within this times R
    int32_t *out_draw;     // nullable [B][4]: fp32 token, listed, exact token, reserved
    int B, k, V;
    int NS;            // tiles per row
    int NSS;           // super-tiles per row
    int rows;          // rows per sequence (2k+1)
    int DS;            // draw tiles per row
    int chunk_stride;  // floats of chunk totals per sequence
    int NCH;           // 4 KB chunks per row
    unsigned int total_super;  // super-tiles in the call
    unsigned long long target_bytes, draft_bytes;
};

struct Smem {
    unsigned long long full[STAGES];
    unsigned long long empty[STAGES];
    TileInfo info[STAGES];
    float4 wpart[STAGES][NCW];
    int wcnt[STAGES];
};

constexpr size_t SMEM_BYTES = (size_t)STAGES * SLOT_BYTES + sizeof(Smem);

// ------------------------------------------------------------ row statistics
//
// Lane state over one super-tile: running maximum m, sum s of 2^((x-m)*c)
// relative to it (sampling), lowest index attaining it (greedy).  Consumer
// thread t owns vectors t, t+NT, ... of every tile.

struct LaneStat {
    float m, s;
    int idx;
};

// Consumer warp w owns the contiguous 4 KB chunk w of a tile: lane l reads the
// tile's vectors 256*w + 32*u + l, u < U.  `rec` (nullable) receives the
// chunk's record (maximum, sum of 2^((x - max) * c)) on a bonus row; `gk`
// (nullable, the warp's 32 slots) the order key of the maximum of each lane's
// U vectors, for the top-k cut of a filtered call.
template <int DT>
__device__ __forceinline__ void tile_accumulate(const Seg &g, int warp, int lane, int mode, float c,
                                                LaneStat &st, float2 *rec, unsigned int *gk)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    const int v0 = g.e0 / VEC;
    const int v1 = (g.e1 + VEC - 1) / VEC;
    const int base = warp * 32 * U + lane;  // tile-relative vector of u = 0

    uint4 raw[U];
    if (g.fast && g.e1 - g.e0 == U * NT * VEC) {
        // a whole tile, copied aligned: every vector is in range
#pragma unroll
        for (int u = 0; u < U; ++u)
            raw[u] = ld_shared_v4(g.slot + (size_t)(base + u * 32) * 16);
    } else {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + base + u * 32;
            raw[u] = (v < v1) ? seg_vec<DT>(g, v) : neg_inf_vec(L::NEG_INF_WORD);
        }
    }

    if (mode == MODE_GREEDY) {
        float vmax[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            vmax[u] = L::vmax(raw[u]);
        float mt = vmax[0];
#pragma unroll
        for (int u = 1; u < U; ++u)
            mt = fmax_nan(mt, vmax[u]);
        if (gk)
            __stcg(gk + lane, key_of<DT>(mt));
        // the lane's indices grow with u, and the first occurrence over the
        // super-tile lies in the earliest tile holding a strictly larger maximum
        if (mt > st.m) {
            int idx = INT_MAX;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (idx == INT_MAX && vmax[u] == mt) {
                    float x[VEC];
                    L::unpack(raw[u], x);
#pragma unroll
                    for (int j = VEC - 1; j >= 0; --j)
                        if (x[j] == mt)
                            idx = (v0 + base + u * 32) * VEC + j;
                }
            }
            st.idx = idx;
        }
        st.m = fmax_nan(st.m, mt);
        return;
    }
    // sampling: the tile's sum against the lane's tile maximum, folded into the
    // running (m, s) with one rescale of each side
    const float mt = L::tile_max(raw);
    if (gk)
        __stcg(gk + lane, key_of<DT>(mt));
    float ts = 0.0f;
    if (mt != -INFINITY) {
        const unsigned long long c2 = f2(c, c);
        unsigned long long acc = L::expsum2(raw[0], -mt, c2);
#pragma unroll
        for (int u = 1; u < U; ++u)
            acc = add2(acc, L::expsum2(raw[u], -mt, c2));
        float s0, s1;
        f2_split(acc, s0, s1);
        ts = s0 + s1;
    }
    const float mn = fmax_nan(st.m, mt);
    if (mn != st.m)
        st.s = rescale(st.s, st.m, mn, c);
    st.s += (mt == mn) ? ts : rescale(ts, mt, mn, c);
    st.m = mn;
    if (rec) {
        float M = mt;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            M = fmax_nan(M, __shfl_xor_sync(0xffffffffu, M, o));
        float S = (mt == M) ? ts : rescale(ts, mt, M, c);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            S += __shfl_xor_sync(0xffffffffu, S, o);
        if (lane == 0)
            __stcg(rec, make_float2(M, S));
    }
}

template <int DT>
__global__ void __launch_bounds__(NTHREADS, 2) stats_kernel(const Params P)
{
    using L = Lg<DT>;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *slots = smem_raw;
    Smem &S = *reinterpret_cast<Smem *>(smem_raw + (size_t)STAGES * SLOT_BYTES);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    constexpr int SEG = TILE_BYTES / L::ES;

    if (tid == 0) {
        if (blockIdx.x == 0) {  // later kernels' counters (they run after this grid)
            P.hdr->next_item = 0u;
            P.hdr->next_item2 = 0u;
            P.hdr->n_flag = 0u;
            P.hdr->next_resolve = 0u;
            P.hdr->n_slow_ratio = 0u;
            P.hdr->n_slow_kinks = 0u;
            P.hdr->n_stream_rows = 0u;
            P.hdr->n_radix_rows = 0u;
            P.hdr->n_stream_draws = 0u;
        }
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], NCW);
            S.wcnt[s] = 0;
        }
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
        bool ok = true;
        const unsigned int supers_per_seq = (unsigned int)P.rows * (unsigned int)P.NSS;
        // super-tiles are dealt round robin: CTA i takes i, i+G, i+2G, ...
        for (unsigned int st = blockIdx.x; st < P.total_super && ok; st += gridDim.x) {
            const int b = (int)(st / supers_per_seq);
            const unsigned int rem = st - (unsigned int)b * supers_per_seq;
            const int rsq = (int)(rem / (unsigned int)P.NSS);
            const int sst = (int)(rem - (unsigned int)rsq * (unsigned int)P.NSS);
            const float T = __ldg(P.temperature + b);
            int mode;
            if (!temperature_valid(T))
                mode = MODE_SKIP;
            else if (T == 0.0f)
                mode = (rsq <= P.k) ? MODE_GREEDY : MODE_SKIP;  // greedy never reads drafts
            else
                mode = MODE_SAMPLE;
            if (mode == MODE_SKIP)
                continue;  // nobody reads this row's statistics
            const bool is_target = rsq <= P.k;
            const uint8_t *arr = reinterpret_cast<const uint8_t *>(is_target ? P.target : P.draft);
            const unsigned long long arr_bytes = is_target ? P.target_bytes : P.draft_bytes;
            const unsigned long long row = is_target ? (unsigned long long)b * (P.k + 1) + rsq
                                                     : (unsigned long long)b * P.k + (rsq - P.k - 1);
            const int seg0 = sst * SUPER;
            const int seg1 = min(P.NS, seg0 + SUPER);
            for (int seg = seg0; seg < seg1; ++seg) {
                if (!mbar_wait(&S.empty[stage], phase ^ 1u)) {
                    atomicExch(&P.hdr->status, SPEC_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                TileInfo &ti = S.info[stage];
                ti.kind = KIND_STATS;
                ti.b = b;
                ti.rsq = rsq;
                ti.seg = seg;
                ti.mode = mode;
                ti.last = (seg == seg1 - 1) ? 1 : 0;
                ti.c = (mode == MODE_SAMPLE) ? LOG2E / T : 0.0f;
                ti.bonus = (mode == MODE_SAMPLE && rsq == P.k) ? 1 : 0;
                const int e0 = seg * SEG, e1 = min(P.V, e0 + SEG);
                const unsigned long long start = (row * P.V + e0) * L::ES;
                const unsigned long long end = (row * P.V + e1) * L::ES;
                const unsigned long long a0 = start & ~15ull;
                unsigned long long a1 = (end + 15) & ~15ull;
                if (a1 > (arr_bytes & ~15ull))
                    a1 = arr_bytes & ~15ull;
                const uint32_t bytes = (a1 > a0) ? (uint32_t)(a1 - a0) : 0u;
                ti.phase0 = (int)(start - a0);
                ti.ncopied0 = (int)bytes;
                if (bytes) {
                    mbar_arrive_expect_tx(&S.full[stage], bytes);
                    bulk_copy_g2s(slots + (size_t)stage * SLOT_BYTES, arr + a0, bytes, &S.full[stage]);
                } else {
                    mbar_arrive(&S.full[stage]);
                }
                issued_phase[stage] = (int)phase;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (ok) {
            if (mbar_wait(&S.empty[stage], phase ^ 1u)) {
                S.info[stage].kind = KIND_END;
                mbar_arrive(&S.full[stage]);
            } else {
                atomicExch(&P.hdr->status, SPEC_DEV_WAIT_TIMEOUT);
                ok = false;
            }
        }
        if (!ok) {
            // let the copies already issued land before leaving
            for (int s = 0; s < STAGES; ++s)
                if (issued_phase[s] >= 0)
                    (void)mbar_wait(&S.full[s], (uint32_t)issued_phase[s]);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    int stage = 0;
    uint32_t phase = 0;
    LaneStat st = {-INFINITY, 0.0f, INT_MAX};
    while (true) {
        if (!mbar_wait(&S.full[stage], phase)) {
            if (lane == 0)
                atomicExch(&P.hdr->status, SPEC_DEV_WAIT_TIMEOUT);
            break;
        }
        const TileInfo ti = S.info[stage];
        if (ti.kind == KIND_END)
            break;
        const uint8_t *slot = slots + (size_t)stage * SLOT_BYTES;
        const bool is_target = ti.rsq <= P.k;
        const size_t row = is_target ? (size_t)ti.b * (P.k + 1) + ti.rsq
                                     : (size_t)ti.b * P.k + (ti.rsq - P.k - 1);
        const int e0 = ti.seg * SEG, e1 = min(P.V, e0 + SEG);
        const Seg g = make_seg<DT>(slot, is_target ? P.target : P.draft, row, P.V, e0, e1, ti.phase0,
                                   ti.ncopied0);
        float2 *rec = nullptr;
        if (ti.bonus) {
            const int q = ti.seg * NCW + warp;  // 4 KB chunk of the bonus row
            if (q < P.NCH)
                rec = P.rec + (size_t)ti.b * P.NCH + q;
        }
        unsigned int *gk = P.gkey ? P.gkey + ((size_t)ti.b * P.rows + ti.rsq) * (size_t)P.NS * NT +
                                        (size_t)ti.seg * NT + (size_t)warp * 32
                                  : nullptr;
        tile_accumulate<DT>(g, warp, lane, ti.mode, ti.c, st, rec, gk);
        if (!ti.last) {
            // the slot is free once every warp has read it
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&S.empty[stage]);
        } else {
            // end of a super-tile: warp, then CTA combine into one partial
            float m = st.m, s = st.s;
            int idx = st.idx;
            warp_combine(m, s, idx, ti.c, ti.mode == MODE_SAMPLE);
            st.m = -INFINITY;
            st.s = 0.0f;
            st.idx = INT_MAX;
            if (lane == 0)
                S.wpart[stage][warp] = make_float4(m, s, __int_as_float(idx), 0.0f);
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                last = (atomicAdd_block(&S.wcnt[stage], 1) == NCW - 1) ? 1 : 0;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence_block();
                float m2 = -INFINITY, s2 = 0.0f;
                int i2 = INT_MAX;
                if (lane < NCW) {
                    const float4 r = S.wpart[stage][lane];
                    m2 = r.x;
                    s2 = r.y;
                    i2 = __float_as_int(r.z);
                }
                warp_combine(m2, s2, i2, ti.c, ti.mode == MODE_SAMPLE);
                if (lane == 0) {
                    __stcg(P.part + ((size_t)ti.b * P.rows + ti.rsq) * P.NSS + ti.seg / SUPER,
                           make_float4(m2, s2, __int_as_float(i2), 0.0f));
                    S.wcnt[stage] = 0;
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&S.empty[stage]);
        }
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

// ---------------------------------------------------- top-k / top-p filter
//
// One CTA per row of every sequence whose call asks for filtering.  The kept
// set is a prefix of the row ranked by (logit descending, index ascending):
// top-k keeps the first K; top-p keeps, among those, a token while the mass
// ranked before it is below P times the top-k mass.  Its end (the last kept
// token) is found by a radix search on the order-preserving key, four bits per
// pass from the top.  Each pass reads the row (from L2 after the first) and
// fills per-thread columns of a shared-memory histogram -- counts, and masses
// 2^((x - m) * c) in 2^-40 fixed point -- that are summed in a fixed order, so
// every decision is deterministic.  As soon as the bucket holding the end has
// at most FCAP tokens, they are gathered in index order, sorted by (key desc,
// index asc) and the end is read off the sorted list; if a single key value
// holds more ties than that, a pass in index order counts them instead.

constexpr int FTH = 256;         // filter threads
constexpr int FBINS = 16;        // buckets per pass (4-bit digits)
constexpr int WBINS = 64;        // half-bit distance bins of the one-pass window
static_assert(WBINS == 64, "the window statistics give each lane of a warp two bins");
constexpr int FCAP = 1024;       // tokens finished by a sort in shared memory
constexpr int FSLOTS = 4;        // ring slots of a row pass
constexpr int FTILE = 16384;     // bytes of a row per slot
constexpr int FSLOT_BYTES = FTILE + 128;  // room for a misaligned head/tail
constexpr int FVPT = FTILE / (16 * 256);  // 16-byte vectors per thread per tile
constexpr float FIX = 1099511627776.0f;  // 2^40

struct FiltTile {
    int e0, e1, phase0, ncopied;
};

struct FiltSmem {
    uint8_t ring[FSLOTS][FSLOT_BYTES];  // a row pass streams through these
    unsigned long long fbar[FSLOTS];
    FiltTile tile[FSLOTS];
    int waitok;
    union __align__(16) {  // 16-byte aligned: the histogram is zeroed with uint4 stores
        struct {
            struct {
                unsigned long long key[FCAP];  // (key << 32) | ~index: descending = the ranking
                unsigned long long mass[FCAP];
            } c;  // gathered tokens (any order), sorted in place by bitonic
            struct {
                unsigned long long key[FCAP];
                unsigned long long mass[FCAP];
            } r;  // rank placement's output, or the window's second buffer
        } cr;
        struct {
            unsigned int cnt[4][FBINS][32];  // a column per lane: no two lanes of a
            unsigned long long mass[4][FBINS][32];  // warp add to one word (warps w, w+4 share)
        } h;  // the general case's histogram (not live while tokens are gathered)
    } u;
    unsigned int ncand;                 // tokens gathered so far
    unsigned int fh_cnt[WBINS];         // window histogram: tokens per half-bit bin
    unsigned long long fh_mass[WBINS];  // and their masses (integer atomics)
    int wnb;                            // window bin limit / bin of the cut
    unsigned int wcum;                  // tokens through the cut's bin
    int whalf;                          // last bin holding at most FCAP / 2 tokens through it
    unsigned int bcnt[FBINS];
    unsigned long long bmass[FBINS];
    unsigned int wcnt[FTH / 32];
    unsigned long long wmass[FTH / 32];
    float m;
    int flags;
    int sel;                 // selected bucket, or -1
    int found;               // index found by a tie pass
    unsigned long long acc;  // scratch sum
};
constexpr size_t FILT_SMEM = sizeof(FiltSmem);
static_assert(FVPT * 16 * FTH == FTILE, "a filter tile splits evenly over the threads");
static_assert(FTH == 16 * FBINS && FTH / 32 == 8, "the histogram reduction's thread map");
static_assert(offsetof(FiltSmem, u) % 16 == 0 && sizeof(FiltSmem::u) % 16 == 0,
              "the sort / histogram union takes uint4 stores");

__device__ __forceinline__ unsigned long long fixmass(float x, float m, float c)
{
    return __float2ull_rn(ex2((x - m) * c) * FIX);
}

// A slot in the sort buffer for every lane with `want`, one shared atomic per
// warp; the whole warp must call it.
__device__ __forceinline__ unsigned int warp_slot(bool want, unsigned int *counter, int lane)
{
    const unsigned int mask = __ballot_sync(0xffffffffu, want);
    unsigned int base = 0u;
    if (mask && lane == __ffs(mask) - 1)
        base = atomicAdd(counter, (unsigned int)__popc(mask));
    base = __shfl_sync(0xffffffffu, base, mask ? __ffs(mask) - 1 : 0);
    return base + (unsigned int)__popc(mask & ((1u << lane) - 1u));
}

__device__ __forceinline__ unsigned long long sortkey(unsigned int key, int idx)
{
    return ((unsigned long long)key << 32) | (unsigned long long)(0xffffffffu - (unsigned int)idx);
}

// Block-wide exclusive prefix of one count per thread (index order = thread
// order) and the block total.
__device__ __forceinline__ unsigned int block_excl_scan(unsigned int x, FiltSmem &S,
                                                        unsigned int &total)
{
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    unsigned int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        S.wcnt[warp] = incl;
    __syncthreads();
    unsigned int wbase = 0, tot = 0;
    for (int w = 0; w < FTH / 32; ++w) {
        const unsigned int v = S.wcnt[w];
        if (w < warp)
            wbase += v;
        tot += v;
    }
    __syncthreads();
    total = tot;
    return wbase + incl - x;
}

template <int DT>
__global__ void __launch_bounds__(FTH, 2) filter_kernel(const Params P)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    constexpr int LOW_SHIFT = (DT == SPEC_F32) ? 0 : 16;  // bf16 keys end at bit 16
    extern __shared__ __align__(16) uint8_t fsm_raw[];
    FiltSmem &S = *reinterpret_cast<FiltSmem *>(fsm_raw);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int V = P.V;
    const int items = P.B * P.rows;
    if (t == 0) {
        for (int q = 0; q < FSLOTS; ++q)
            mbar_init(&S.fbar[q], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    unsigned int par = 0u;  // completed-phase parity of each ring slot (same in every thread)
    bool failed = false;    // a bulk copy never landed: stop this CTA
    allow_next_kernel();
    wait_previous_kernel();  // partials come from the statistics kernel
    if (__ldcg(&P.hdr->n_radix_rows) == 0u)
        return;  // no row was left to the radix search

    // This kernel finishes the rows the window kernel recorded FILT_RADIX
    // (its buffer overflowed, or its window ended short of the cut).  Rows
    // are taken in chunks of up to 32 from the second header counter (zeroed
    // by the statistics kernel), small enough that each CTA gets several;
    // a chunk's flags are read by one warp.
    const int chunk = max(1, min(32, items / ((int)gridDim.x * 8)));
    unsigned int fmask = 0u;
    int fbase = 0;
    auto next_item = [&]() -> int {
        for (;;) {
            if (fmask) {
                const int i = __ffs(fmask) - 1;
                fmask &= fmask - 1u;
                return fbase + i;
            }
            __syncthreads();
            if (t == 0)
                S.found = (int)atomicAdd(&P.hdr->next_item2, (unsigned int)chunk);
            __syncthreads();
            fbase = S.found;
            if (fbase >= items)
                return items;
            if (warp == 0) {
                const int it = fbase + lane;
                const bool f = lane < chunk && it < items &&
                               __ldcg(&P.filt[it].flags) == FILT_RADIX;
                const unsigned int bm = __ballot_sync(0xffffffffu, f);
                if (lane == 0)
                    S.sel = (int)bm;
            }
            __syncthreads();
            fmask = (unsigned int)S.sel;
        }
    };
    for (int item = next_item(); item < items && !failed; item = next_item()) {
        const int b = item / P.rows, rsq = item - b * P.rows;
        const bool is_target = rsq <= P.k;
        const void *arr = is_target ? P.target : P.draft;
        const size_t row = is_target ? (size_t)b * (P.k + 1) + rsq
                                     : (size_t)b * P.k + (rsq - P.k - 1);
        const float T = __ldg(P.temperature + b);
        const int K = P.top_k ? __ldg(P.top_k + b) : 0;
        const float Pp = P.top_p ? __ldg(P.top_p + b) : 1.0f;
        FiltRec out;
        out.kappa = 0u;
        out.iota = INT_MAX;
        out.zt = 0.0f;
        out.flags = FILT_OFF;
        const bool topk = K > 0 && K < V;
        const bool topp = Pp < 1.0f;
        const bool bad = K < 0 || isnan(Pp) || !(Pp > 0.0f);
        if (temperature_valid(T) && bad) {
            out.flags = FILT_ERR;  // bad filter parameters fail the sequence, greedy too
            if (t == 0)
                P.filt[item] = out;
            continue;
        }
        if (!temperature_valid(T) || T == 0.0f || (!topk && !topp)) {
            if (t == 0)
                P.filt[item] = out;  // greedy, invalid or unfiltered: nothing to keep out
            continue;
        }
        // the row maximum and total mass from the statistics kernel's partials
        const float c = LOG2E / T;
        if (warp == 0) {
            const float4 *pp = P.part + ((size_t)b * P.rows + rsq) * P.NSS;
            float m = -INFINITY;
            for (int q = lane; q < P.NSS; q += 32)
                m = fmax_nan(m, __ldcg(pp + q).x);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
            float z = 0.0f;
            for (int q = lane; q < P.NSS; q += 32) {
                const float4 pv = __ldcg(pp + q);
                z += rescale(pv.y, pv.x, m, c);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                z += __shfl_xor_sync(0xffffffffu, z, o);
            if (lane == 0) {
                S.m = m;
                S.acc = (unsigned long long)((double)z * 1099511627776.0);
            }
        }
        __syncthreads();
        const float m = S.m;
        const unsigned long long Zrow = S.acc;  // 2^-40 fixed point
        __syncthreads();
        if (isnan(m) || isinf(m)) {
            if (t == 0)
                P.filt[item] = out;  // the scan reports the row as an error
            continue;
        }

        // A row pass streams the row through the ring: thread 0 keeps up to
        // FSLOTS 16 KB bulk copies in flight; every thread reads its FVPT
        // vectors of each tile from shared memory (thread t: vectors
        // t + q * FTH of the tile).  Waits are decided by thread 0 and shared,
        // so every thread takes the same path; a copy that never lands
        // (bounded wait) stops the CTA with SPEC_DEV_WAIT_TIMEOUT.
        constexpr int TE = FTILE / L::ES;  // elements per tile
        const int ntiles = (V + TE - 1) / TE;
        const unsigned long long arr_bytes = is_target ? P.target_bytes : P.draft_bytes;
        auto issue = [&](int i) {  // thread 0: tile i into slot i % FSLOTS
            const int q = i % FSLOTS;
            const int e0 = i * TE, e1 = min(V, e0 + TE);
            const unsigned long long start = ((unsigned long long)row * V + e0) * L::ES;
            const unsigned long long end = ((unsigned long long)row * V + e1) * L::ES;
            const unsigned long long a0 = start & ~15ull;
            unsigned long long a1 = (end + 15) & ~15ull;
            if (a1 > (arr_bytes & ~15ull))
                a1 = arr_bytes & ~15ull;
            const uint32_t bytes = (a1 > a0) ? (uint32_t)(a1 - a0) : 0u;
            S.tile[q].e0 = e0;
            S.tile[q].e1 = e1;
            S.tile[q].phase0 = (int)(start - a0);
            S.tile[q].ncopied = (int)bytes;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (bytes) {
                mbar_arrive_expect_tx(&S.fbar[q], bytes);
                bulk_copy_g2s(S.ring[q], reinterpret_cast<const uint8_t *>(arr) + a0, bytes,
                              &S.fbar[q]);
            } else {
                mbar_arrive(&S.fbar[q]);
            }
        };
        // fn(raw[FVPT], vt0): the thread's vectors vt0 + q * FTH of one tile
        // after(raw, vt0, e0, e1), if given, runs in every thread once the tile
        // is done and its slot refilled (the thread's vectors are still in raw)
        auto stream_row_then = [&](auto fn, auto after) {
            if (failed)
                return;
            if (t == 0)
                for (int i = 0; i < min(FSLOTS, ntiles); ++i)
                    issue(i);
            for (int i = 0; i < ntiles; ++i) {
                const int q = i % FSLOTS;
                const uint32_t pq = (par >> q) & 1u;
                if (t == 0)
                    S.waitok = mbar_wait(&S.fbar[q], pq) ? 1 : 0;
                __syncthreads();
                if (!S.waitok) {
                    failed = true;
                    if (t == 0) {
                        atomicExch(&P.hdr->status, SPEC_DEV_WAIT_TIMEOUT);
                        // let the other copies in flight land (bounded)
                        for (int i2 = i + 1; i2 < min(i + FSLOTS, ntiles); ++i2)
                            (void)mbar_wait(&S.fbar[i2 % FSLOTS], (par >> (i2 % FSLOTS)) & 1u);
                    }
                    __syncthreads();
                    return;
                }
                (void)mbar_try_wait(&S.fbar[q], pq);  // acquire the landed bytes
                const FiltTile ti = S.tile[q];
                const Seg g = make_seg<DT>(S.ring[q], arr, row, V, ti.e0, ti.e1, ti.phase0,
                                           ti.ncopied);
                const int vt0 = ti.e0 / VEC;
                uint4 raw[FVPT];
                if (g.fast && ti.e1 - ti.e0 == TE) {
#pragma unroll
                    for (int u = 0; u < FVPT; ++u)
                        raw[u] = ld_shared_v4(S.ring[q] + (size_t)(t + u * FTH) * 16);
                } else {
#pragma unroll
                    for (int u = 0; u < FVPT; ++u)
                        raw[u] = seg_vec<DT>(g, vt0 + t + u * FTH);
                }
                fn(raw, vt0);
                __syncthreads();  // every thread is done with slot q
                par ^= 1u << q;
                if (t == 0 && i + FSLOTS < ntiles)
                    issue(i + FSLOTS);
                after(raw, vt0, ti.e0, ti.e1);
            }
        };
        auto stream_row = [&](auto fn) {
            stream_row_then(fn, [](const uint4 (&)[FVPT], int, int, int) {});
        };
        auto member = [](unsigned int key, int idx, unsigned int kk, int ik) {
            return key > kk || (key == kk && idx <= ik);
        };
        // histogram of bin_of(x, key, idx) (-1: not counted): counts and masses
        auto hist = [&](auto bin_of, auto vskip) {
            for (int i = t; i < (int)(sizeof(S.u.h) / 16); i += FTH)
                reinterpret_cast<uint4 *>(&S.u.h)[i] = make_uint4(0u, 0u, 0u, 0u);
            __syncthreads();
            unsigned int *hc = &S.u.h.cnt[warp & 3][0][lane];
            unsigned long long *hm = &S.u.h.mass[warp & 3][0][lane];
            stream_row([&](const uint4 (&r)[FVPT], int vt0) {
#pragma unroll
                for (int u = 0; u < FVPT; ++u) {
                    if (vskip(r[u]))
                        continue;  // no token of this vector can count
                    float x[VEC];
                    L::unpack(r[u], x);
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        const int idx = (vt0 + t + u * FTH) * VEC + j;
                        const int bin = (idx < V) ? bin_of(x[j], key_of<DT>(x[j]), idx) : -1;
                        if (bin >= 0) {
                            atomicAdd(hc + bin * 32, 1u);
                            atomicAdd(hm + bin * 32, fixmass(x[j], m, c));
                        }
                    }
                }
            });
            __syncthreads();
            {  // bin t / 16: sixteen threads sum its 128 columns
                const int bb = t >> 4, part = t & 15;
                unsigned int cs = 0u;
                unsigned long long ms = 0ull;
                for (int q = part; q < 128; q += 16) {
                    cs += S.u.h.cnt[q >> 5][bb][q & 31];
                    ms += S.u.h.mass[q >> 5][bb][q & 31];
                }
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) {
                    cs += __shfl_xor_sync(0xffffffffu, cs, o);
                    ms += __shfl_xor_sync(0xffffffffu, ms, o);
                }
                if (part == 0) {
                    S.bcnt[bb] = cs;
                    S.bmass[bb] = ms;
                }
            }
            __syncthreads();
        };
        // the tokens with pred(x, key, idx) into the sort buffer, in no
        // particular order (the sort key carries the index); returns how many
        // there are, which may exceed FCAP (only the first FCAP are stored)
        auto gather = [&](auto pred, auto vskip) -> int {
            if (t == 0)
                S.ncand = 0u;
            __syncthreads();
            stream_row([&](const uint4 (&r)[FVPT], int vt0) {
#pragma unroll
                for (int u = 0; u < FVPT; ++u) {
                    const bool live = !vskip(r[u]);
                    if (!__any_sync(0xffffffffu, live))
                        continue;
                    float x[VEC];
                    L::unpack(r[u], x);
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        const int idx = (vt0 + t + u * FTH) * VEC + j;
                        const unsigned int key = key_of<DT>(x[j]);
                        const bool take = live && idx < V && pred(x[j], key, idx);
                        const unsigned int pos = warp_slot(take, &S.ncand, lane);
                        if (take && pos < (unsigned int)FCAP) {  // never past the buffer
                            S.u.cr.c.key[pos] = sortkey(key, idx);
                            S.u.cr.c.mass[pos] = fixmass(x[j], m, c);
                        }
                    }
                }
            });
            __syncthreads();
            const int n = (int)S.ncand;
            __syncthreads();
            return n;
        };
        // bitonic sort of the first n gathered tokens, descending
        auto sort_desc = [&](int n) {
            int p2 = 1;
            while (p2 < n)
                p2 <<= 1;
            for (int i = n + t; i < p2; i += FTH) {
                S.u.cr.c.key[i] = 0ull;
                S.u.cr.c.mass[i] = 0ull;
            }
            __syncthreads();
            for (int kk = 2; kk <= p2; kk <<= 1) {
                for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                    for (int i = t; i < p2; i += FTH) {
                        const int ixj = i ^ jj;
                        if (ixj > i) {
                            const unsigned long long a = S.u.cr.c.key[i], bq = S.u.cr.c.key[ixj];
                            const bool desc = (i & kk) == 0;
                            if (desc ? (a < bq) : (a > bq)) {
                                S.u.cr.c.key[i] = bq;
                                S.u.cr.c.key[ixj] = a;
                                const unsigned long long ma = S.u.cr.c.mass[i];
                                S.u.cr.c.mass[i] = S.u.cr.c.mass[ixj];
                                S.u.cr.c.mass[ixj] = ma;
                            }
                        }
                    }
                    __syncthreads();
                }
            }
        };
        // the sorted list: S.c after a bitonic sort, S.r after rank placement
        unsigned long long *skey = S.u.cr.c.key, *smass = S.u.cr.c.mass;
        // rank placement of n <= FCAP gathered tokens (keys are unique): the
        // rank of a token is the number of larger keys; from one buffer into
        // the other
        auto rank_sort = [&](int n, unsigned long long *ikey, unsigned long long *imass,
                             unsigned long long *okey_, unsigned long long *omass) {
            constexpr int PER = FCAP / FTH;
            unsigned long long mine[PER];
            int rk[PER];
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int i = t + q * FTH;
                mine[q] = (i < n) ? ikey[i] : 0ull;
                rk[q] = 0;
            }
            for (int jj = 0; jj < n; ++jj) {
                const unsigned long long kj = ikey[jj];
#pragma unroll
                for (int q = 0; q < PER; ++q)
                    rk[q] += (kj > mine[q]) ? 1 : 0;
            }
            unsigned long long mm[PER];
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int i = t + q * FTH;
                mm[q] = (i < n) ? imass[i] : 0ull;
            }
            __syncthreads();  // the output may overlap nothing the others still read
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int i = t + q * FTH;
                if (i < n) {
                    okey_[rk[q]] = mine[q];
                    omass[rk[q]] = mm[q];
                }
            }
            __syncthreads();
            skey = okey_;
            smass = omass;
        };
        // sort the n tokens gathered in S.c (from_r: in S.r) into descending order
        auto sort_any = [&](int n, bool from_r = false) {
            if (n <= FCAP / 2) {
                if (from_r)
                    rank_sort(n, S.u.cr.r.key, S.u.cr.r.mass, S.u.cr.c.key, S.u.cr.c.mass);
                else
                    rank_sort(n, S.u.cr.c.key, S.u.cr.c.mass, S.u.cr.r.key, S.u.cr.r.mass);
            } else {
                if (from_r) {
                    for (int i = t; i < n; i += FTH) {
                        S.u.cr.c.key[i] = S.u.cr.r.key[i];
                        S.u.cr.c.mass[i] = S.u.cr.r.mass[i];
                    }
                    __syncthreads();
                }
                sort_desc(n);
                skey = S.u.cr.c.key;
                smass = S.u.cr.c.mass;
            }
        };
        // mass of the first r sorted tokens (fixed order)
        auto sorted_prefix_mass = [&](int r) -> unsigned long long {
            if (warp == 0) {
                unsigned long long ms = 0ull;
                for (int i = lane; i < r; i += 32)
                    ms += smass[i];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    ms += __shfl_xor_sync(0xffffffffu, ms, o);
                if (lane == 0)
                    S.acc = ms;
            }
            __syncthreads();
            const unsigned long long v = S.acc;
            __syncthreads();
            return v;
        };
        // the first of the first n sorted tokens whose running mass (from
        // `start`) reaches the target; its position and that running mass
        auto sorted_cut = [&](int n, unsigned long long start, unsigned long long target,
                              unsigned long long &run_out) -> int {
            if (warp == 0) {
                unsigned long long run = start;
                int istar = -1;
                for (int i0 = 0; i0 < n && istar < 0; i0 += 32) {
                    const int i = i0 + lane;
                    unsigned long long x = (i < n) ? smass[i] : 0ull;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
                        if (lane >= o)
                            x += y;
                    }
                    const unsigned long long incl = run + x;
                    const unsigned hit = __ballot_sync(0xffffffffu, i < n && incl >= target);
                    if (hit) {
                        const int hl = __ffs(hit) - 1;
                        istar = i0 + hl;
                        run = __shfl_sync(0xffffffffu, incl, hl);
                    } else {
                        run = __shfl_sync(0xffffffffu, incl, 31);
                    }
                }
                if (istar < 0)
                    istar = n - 1;  // rounding: all of them
                if (lane == 0) {
                    S.sel = istar;
                    S.acc = run;
                }
            }
            __syncthreads();
            const int i = S.sel;
            run_out = S.acc;
            __syncthreads();
            return i;
        };
        auto sorted_at = [&](int i, unsigned int &key, int &idx) {
            const unsigned long long e = skey[i];
            key = (unsigned int)(e >> 32);
            idx = (int)(0xffffffffu - (unsigned int)(e & 0xffffffffu));
        };
        // the r-th (1-based) token in index order with key == kap (restricted)
        auto tie_pass = [&](unsigned int kap, unsigned int r, bool rk, unsigned int kK,
                            int iK) -> int {
            if (t == 0)
                S.found = -1;
            __syncthreads();
            unsigned int base = 0u;
            stream_row([&](const uint4 (&r4)[FVPT], int vt0) {
                // round u covers vectors vt0 + u*FTH .. +FTH-1: thread order is index order
#pragma unroll
                for (int u = 0; u < FVPT; ++u) {
                    float x[VEC];
                    L::unpack(r4[u], x);
                    const int v = vt0 + t + u * FTH;
                    unsigned int n = 0u;
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        const int idx = v * VEC + j;
                        const unsigned int key = key_of<DT>(x[j]);
                        n += (idx < V && key == kap && (!rk || member(key, idx, kK, iK))) ? 1u : 0u;
                    }
                    unsigned int tot;
                    const unsigned int ex = base + block_excl_scan(n, S, tot);
                    if (n && ex < r && r <= ex + n) {
                        unsigned int cnt = ex;
#pragma unroll
                        for (int j = 0; j < VEC; ++j) {
                            const int idx = v * VEC + j;
                            const unsigned int key = key_of<DT>(x[j]);
                            if (idx < V && key == kap && (!rk || member(key, idx, kK, iK))) {
                                if (++cnt == r)
                                    S.found = idx;
                            }
                        }
                    }
                    base += tot;
                }
            });
            __syncthreads();
            return S.found;
        };
        auto val_of_key = [&](unsigned int key) {
            unsigned int bits = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
            if (DT == SPEC_BF16)
                bits &= 0xffff0000u;
            return __uint_as_float(bits);
        };
        auto fix_of_key = [&](unsigned int key) {
            unsigned int bits = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
            if (DT == SPEC_BF16)
                bits &= 0xffff0000u;
            return fixmass(__uint_as_float(bits), m, c);
        };

        unsigned int kap = 0u;
        int iota = INT_MAX;
        unsigned long long Zt = 0ull;
        auto vnone = [](const uint4 &) { return false; };

        const unsigned long long Ztot = Zrow;
        const unsigned long long target0 =
            topk ? 0ull : (unsigned long long)((double)Pp * (double)Ztot);
        bool done = false;

        // ---- one pass, an adaptive window.  A token's distance below the row
        // maximum, in bits of probability, is dd = (m - x) * log2(e) / T; its
        // window bin is floor(2 dd) (half-bit bins, WBINS of them: 32 bits,
        // past which a token's fixed-point mass is zero).  The pass gathers
        // every token whose bin is at most nbw into the sort buffer and counts
        // them per bin (with their masses when top-p stands alone).  A bin set
        // {0..b} is a prefix of the ranking, so once the counts (masses)
        // through some bin b reach K (P times the row mass) the cut lies
        // among the gathered tokens of bins 0..b, and the window narrows to
        // that bin after each tile.  When the buffer overflows in a tile, the
        // window narrows the same way (or, before the counts reach the cut,
        // to the widest set holding at most FCAP / 2 tokens), the buffer is
        // compacted to it, and the tile's own tokens -- of which some were not
        // stored -- are gathered again.  A row whose cut the window cannot
        // hold (cut bin too crowded, or deeper than 32 bits) takes the radix
        // search.
        auto wbin = [&](float x) {
            const float dd = (m - x) * c;
            return (dd < (float)(WBINS / 2)) ? (int)(dd * 2.0f) : WBINS;
        };
        auto wbin_of_entry = [&](unsigned long long e) { return wbin(val_of_key((unsigned int)(e >> 32))); };
        auto idx_of_entry = [](unsigned long long e) {
            return (int)(0xffffffffu - (unsigned int)(e & 0xffffffffull));
        };
        // the n entries of (ik, im) with keep(entry) into (ok, om), in
        // order; returns how many (every thread)
        auto compact = [&](const unsigned long long *ik, const unsigned long long *im, int n,
                           unsigned long long *ok, unsigned long long *om, auto keep) -> int {
            constexpr int PER = FCAP / FTH;
            bool kp[PER];
            unsigned int cnt = 0u;
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int i = t * PER + q;
                kp[q] = i < n && keep(ik[i]);
                cnt += kp[q] ? 1u : 0u;
            }
            unsigned int total;
            unsigned int o = block_excl_scan(cnt, S, total);
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int i = t * PER + q;
                if (kp[q]) {
                    ok[o] = ik[i];
                    om[o] = im[i];
                    ++o;
                }
            }
            __syncthreads();
            return (int)total;
        };
        const bool need_mass = !topk;
        // The first window: fewer than Z * 2^D tokens lie within D bits (each
        // weighs more than 2^-D of the maximum's), so D = log2(FCAP / Z) bits
        // surely fit; 8 more bits usually still fit and usually hold the cut.
        // If that window ends without the cut and never overflowed, the pass
        // runs once more over all WBINS bins.
        const float zrow = (float)((double)Zrow * (1.0 / 1099511627776.0));
        const int Dg = (int)floorf(log2f((float)FCAP / (fmaxf(zrow, 1.0f) * 1.01f))) + 8;
        int nbw0 = 2 * min(WBINS / 2, max(1, Dg)) - 1;
        int nbw = nbw0;        // the window: bins 0..nbw
        bool overflowed = false;
        unsigned int last_nc = 0u;
        unsigned long long *wk = S.u.cr.c.key, *wm = S.u.cr.c.mass;  // the buffer holding it
        unsigned long long *xk = S.u.cr.r.key, *xm = S.u.cr.r.mass;  // the other one
        const unsigned int kmin = topk ? (unsigned int)K : 1u;
        // gather the thread's tokens of one tile within the window (counted
        // in the histogram unless `recount` is false)
        // Each lane marks its tokens of the tile inside the window (no warp
        // collective per token: most vectors hold none), the warp reserves
        // their slots with one scan and one atomic, and only marked tokens
        // are written (and counted in the histogram unless `recount` is
        // false).
        auto gather_window = [&](const uint4 (&r)[FVPT], int vt0, bool recount) {
            uint32_t tb[FVPT];
            unsigned int cnt = 0u;
#pragma unroll
            for (int u = 0; u < FVPT; ++u) {
                tb[u] = 0u;
                if (wbin(L::vmax(r[u])) <= nbw) {  // else no token of the vector is in
                    float x[VEC];
                    L::unpack(r[u], x);
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        const int idx = (vt0 + t + u * FTH) * VEC + j;
                        if (idx < V && wbin(x[j]) <= nbw)
                            tb[u] |= 1u << j;
                    }
                }
                cnt += (unsigned int)__popc(tb[u]);
            }
            unsigned int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += y;
            }
            const unsigned int wtot = __shfl_sync(0xffffffffu, incl, 31);
            if (wtot == 0u)
                return;  // (uniform over the warp)
            unsigned int base = 0u;
            if (lane == 31)
                base = atomicAdd(&S.ncand, wtot);
            unsigned int pos = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
#pragma unroll
            for (int u = 0; u < FVPT; ++u) {
                if (tb[u] == 0u)
                    continue;
                float x[VEC];
                L::unpack(r[u], x);
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    if (!((tb[u] >> j) & 1u))
                        continue;
                    const int idx = (vt0 + t + u * FTH) * VEC + j;
                    const bool keep = pos < (unsigned int)FCAP;  // never past the buffer
                    const unsigned long long e =
                        (keep || (recount && need_mass)) ? fixmass(x[j], m, c) : 0ull;
                    if (recount) {
                        const int wb = wbin(x[j]);
                        atomicAdd(&S.fh_cnt[wb], 1u);
                        if (need_mass)
                            atomicAdd(&S.fh_mass[wb], e);
                    }
                    if (keep) {
                        wk[pos] = sortkey(key_of<DT>(x[j]), idx);
                        wm[pos] = e;
                    }
                    ++pos;
                }
            }
        };
        // warp 0: over the bins 0..nbw, the first bin through which the
        // counts (masses) reach the cut (S.wnb, -1 if none) with the count
        // through it (S.wcum), and the last bin through which at most FCAP / 2
        // tokens lie (S.whalf, -1 if none).  Lane l holds bins 2l and 2l + 1.
        auto window_stats = [&]() {
            const int b0 = 2 * lane, b1 = b0 + 1;
            const unsigned int c0 = (b0 <= nbw) ? S.fh_cnt[b0] : 0u;
            const unsigned int c1 = (b1 <= nbw) ? S.fh_cnt[b1] : 0u;
            const unsigned long long m0 = (b0 <= nbw) ? S.fh_mass[b0] : 0ull;
            const unsigned long long m1 = (b1 <= nbw) ? S.fh_mass[b1] : 0ull;
            unsigned int ci = c0 + c1;
            unsigned long long mi = m0 + m1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned int y = __shfl_up_sync(0xffffffffu, ci, o);
                const unsigned long long ym = __shfl_up_sync(0xffffffffu, mi, o);
                if (lane >= o) {
                    ci += y;
                    mi += ym;
                }
            }
            const unsigned int ce0 = ci - c1;  // through bin b0
            const unsigned long long me0 = mi - m1;
            auto hits = [&](unsigned int cc, unsigned long long mm) {
                return topk ? cc >= (unsigned int)K : mm >= target0;
            };
            const bool h0 = b0 <= nbw && hits(ce0, me0);
            const bool h1 = b1 <= nbw && hits(ci, mi);
            const unsigned int hb = __ballot_sync(0xffffffffu, h0 || h1);
            const unsigned int nh =
                (unsigned int)__popc(__ballot_sync(0xffffffffu, b0 <= nbw && ce0 <= FCAP / 2)) +
                (unsigned int)__popc(__ballot_sync(0xffffffffu, b1 <= nbw && ci <= FCAP / 2));
            if (hb) {
                const int L0 = __ffs(hb) - 1;
                const bool first0 = __shfl_sync(0xffffffffu, h0, L0);
                const unsigned int cb = __shfl_sync(0xffffffffu, first0 ? ce0 : ci, L0);
                if (lane == 0) {
                    S.wnb = first0 ? 2 * L0 : 2 * L0 + 1;
                    S.wcum = cb;
                }
            } else if (lane == 0) {
                S.wnb = -1;
                S.wcum = 0u;
            }
            if (lane == 0)
                S.whalf = (int)nh - 1;
        };
        int bk = -1, ncut = 0, n = 0;
        for (;;) {
            if (t < WBINS) {
                S.fh_cnt[t] = 0u;
                S.fh_mass[t] = 0ull;
            }
            if (t == 0)
                S.ncand = 0u;
            __syncthreads();
            stream_row_then([&](const uint4 (&r)[FVPT], int vt0) { gather_window(r, vt0, true); },
                            [&](const uint4 (&r)[FVPT], int vt0, int e0, int e1) {
                const unsigned int nc = S.ncand;  // (read by every thread after the tile's barrier)
                if (nc <= (unsigned int)FCAP) {
                    // no overflow: once the tokens so far can hold the cut,
                    // narrow the window to the cut's bin (the buffer may keep
                    // tokens past it; they are dropped before the sort).
                    // Checked each time the count has doubled: a few times
                    // a row.
                    if (nc < kmin || nc < 2u * last_nc)
                        return;
                    last_nc = nc;
                    if (warp == 0)
                        window_stats();
                    __syncthreads();
                    if (S.wnb >= 0 && S.wnb < nbw)
                        nbw = S.wnb;
                    __syncthreads();
                    return;
                }
                overflowed = true;
                if (warp == 0)
                    window_stats();
                __syncthreads();
                if (t == 0)
                    S.wnb = (S.wnb >= 0) ? ((S.wcum <= (unsigned int)FCAP) ? S.wnb : -1) : S.whalf;
                __syncthreads();
                nbw = S.wnb;
                // keep the stored tokens of the narrower window, except this
                // tile's, which are gathered again in full
                const int nk = compact(wk, wm, FCAP, xk, xm, [&](unsigned long long en) {
                    const int ix = idx_of_entry(en);
                    return (ix < e0 || ix >= e1) && wbin_of_entry(en) <= nbw;
                });
                unsigned long long *tk_ = wk, *tm_ = wm;
                wk = xk;
                wm = xm;
                xk = tk_;
                xm = tm_;
                if (t == 0)
                    S.ncand = (unsigned int)nk;
                __syncthreads();
                gather_window(r, vt0, false);
                __syncthreads();
            });
            __syncthreads();
            n = (int)S.ncand;  // <= FCAP: every overflow was resolved
            if (warp == 0)
                window_stats();
            __syncthreads();
            bk = S.wnb;
            ncut = (int)S.wcum;
            __syncthreads();
            if (bk >= 0 || failed || overflowed || nbw0 == WBINS - 1)
                break;
            nbw0 = nbw = WBINS - 1;  // the first window was too narrow: all bins
            last_nc = 0u;
            wk = S.u.cr.c.key;
            wm = S.u.cr.c.mass;
            xk = S.u.cr.r.key;
            xm = S.u.cr.r.mass;
        }
        if (bk >= 0 && !failed) {
            if (ncut < n) {  // sort only the bins through the cut's
                n = compact(wk, wm, n, xk, xm,
                            [&](unsigned long long en) { return wbin_of_entry(en) <= bk; });
                wk = xk;
                wm = xm;
            }
            sort_any(n, wk == S.u.cr.r.key);
            const int nk = topk ? K : n;
            const unsigned long long ZK = topk ? sorted_prefix_mass(K) : Ztot;
            int last = nk - 1;
            Zt = ZK;
            if (topp) {
                unsigned long long target = (unsigned long long)((double)Pp * (double)ZK);
                if (target == 0ull)
                    target = 1ull;
                last = sorted_cut(nk, 0ull, target, Zt);
            }
            sorted_at(last, kap, iota);
            done = true;
        }
        if (!done) {
            // ---- general case: radix search on the key, 4 bits per pass
            unsigned int kK = 0u;
            int iK = INT_MAX;
            unsigned long long ZK = Ztot;
            if (topk) {
                unsigned int prefix = 0u, pmask = 0u, above = 0u;
                unsigned long long amass = 0ull;
                for (int shift = 28; shift >= LOW_SHIFT; shift -= 4) {
                    hist([&](float, unsigned int key, int) {
                        return ((key & pmask) == prefix) ? (int)((key >> shift) & (FBINS - 1)) : -1;
                    }, vnone);
                    int sel = 0;
                    for (int bb = FBINS - 1; bb >= 0; --bb) {
                        if (above + S.bcnt[bb] >= (unsigned int)K) {
                            sel = bb;
                            break;
                        }
                        above += S.bcnt[bb];
                        amass += S.bmass[bb];
                    }
                    const unsigned int nsel = S.bcnt[sel];
                    prefix |= (unsigned int)sel << shift;
                    pmask |= (unsigned int)(FBINS - 1) << shift;
                    const unsigned int r = (unsigned int)K - above;
                    if (nsel <= (unsigned int)FCAP) {
                        const int n = gather([&](float, unsigned int key, int) {
                            return (key & pmask) == prefix;
                        }, vnone);
                        sort_any(n);
                        ZK = amass + sorted_prefix_mass((int)r);
                        sorted_at((int)r - 1, kK, iK);
                        break;
                    }
                    if (shift == LOW_SHIFT) {  // one key value with more ties than the buffer
                        kK = prefix;
                        iK = tie_pass(kK, r, false, 0u, INT_MAX);
                        ZK = amass + (unsigned long long)r * fix_of_key(kK);
                    }
                }
            }
            kap = kK;
            iota = iK;
            Zt = ZK;
            if (topp) {
                unsigned int prefix = 0u, pmask = 0u;
                unsigned long long amass = 0ull;
                unsigned long long target = (unsigned long long)((double)Pp * (double)ZK);
                if (target == 0ull)
                    target = 1ull;
                for (int shift = 28; shift >= LOW_SHIFT; shift -= 4) {
                    hist([&](float, unsigned int key, int idx) {
                        return ((key & pmask) == prefix && (!topk || member(key, idx, kK, iK)))
                                   ? (int)((key >> shift) & (FBINS - 1))
                                   : -1;
                    }, vnone);
                    int sel = -1;
                    for (int bb = FBINS - 1; bb >= 0; --bb) {
                        if (amass + S.bmass[bb] >= target) {
                            sel = bb;
                            break;
                        }
                        amass += S.bmass[bb];
                    }
                    if (sel < 0)
                        break;  // rounding: the whole top-k set stays
                    const unsigned int nsel = S.bcnt[sel];
                    prefix |= (unsigned int)sel << shift;
                    pmask |= (unsigned int)(FBINS - 1) << shift;
                    if (nsel <= (unsigned int)FCAP) {
                        const int n = gather([&](float, unsigned int key, int idx) {
                            return (key & pmask) == prefix && (!topk || member(key, idx, kK, iK));
                        }, vnone);
                        sort_any(n);
                        const int last = sorted_cut(n, amass, target, Zt);
                        sorted_at(last, kap, iota);
                        break;
                    }
                    if (shift == LOW_SHIFT) {  // ties at one key value: keep r, in index order
                        const unsigned long long e = fix_of_key(prefix);
                        unsigned long long r = (target - amass + e - 1) / e;
                        if (r < 1ull)
                            r = 1ull;
                        if (r > nsel)
                            r = nsel;
                        kap = prefix;
                        iota = tie_pass(kap, (unsigned int)r, topk, kK, iK);
                        Zt = amass + r * e;
                    }
                }
            }
        }
        if (t == 0) {
            out.kappa = kap;
            out.iota = iota;
            out.zt = (float)((double)Zt * (1.0 / 1099511627776.0));
            out.flags = FILT_ON;
            P.filt[item] = out;
        }
        __syncthreads();
    }
}

// ------------------------------------------- top-k: the cut from group maxima
//
// In a filtered call whose workspace has room for them, the statistics kernel
// leaves, per row, the order key of the maximum of each lane's 8 vectors of
// each tile (64 logits of bf16, 32 of fp32): a group.  For a row with top-k,
// K <= KF_KMAX, the K-th largest group key tau is at most the key of the
// row's K-th largest logit (K groups have a maximum >= tau, each of them a
// logit >= tau), so every kept token lies in a group whose key is >= tau.
// Only those groups are read again: their logits with key >= tau are
// gathered, ordered by (key desc, index asc) -- each token's rank is the
// number of larger keys -- and the cut is read off that order exactly as the
// window kernel reads it off its sorted window
// (top-k mass, then the top-p end by the fixed-point masses).  tau is found
// by a radix search over the row's group keys, 8 bits per pass (two passes
// for bf16 keys, whose low 16 bits are zero).  A row with more selected
// groups or gathered tokens than the buffers hold (many ties at tau) is left
// to the radix kernel (FILT_RADIX).  The window kernel skips these rows.
// The kept set of every row cut here is stored in rank order for the
// kept-set draw, which would otherwise gather it again.
constexpr int KF_TH = 128;
constexpr int KF_KMAX = 256;
constexpr int KF_GCAP = 512;   // selected groups at most
constexpr int KF_CAP = 512;    // gathered tokens at most
constexpr int KF_LB = 8;       // group-key loads in flight per thread
constexpr int KF_GB = 1;       // row vectors in flight per thread while gathering
static_assert(KF_KMAX <= KF_CAP && KF_CAP <= KF_GCAP,
              "the kept set fits the buffer, and the group list holds its order");

// The rows the group-maximum cut takes (the same test in the window kernel).
__device__ __forceinline__ bool kf_row(const Params &P, float T, int K, float Pp)
{
    const bool bad = K < 0 || isnan(Pp) || !(Pp > 0.0f);
    return P.gkey != nullptr && temperature_valid(T) && T > 0.0f && !bad && K > 0 && K < P.V &&
           K <= KF_KMAX;
}

struct KfSmem {
    unsigned long long key[KF_CAP], mass[KF_CAP];  // gathered tokens, in gathering order
    int glist[KF_GCAP];                            // selected groups, then the tokens' order
    unsigned int hist[256];
    unsigned int ng, nc;
    unsigned int sel, need;
    unsigned long long red[KF_TH / 32];
};

template <int DT>
__global__ void __launch_bounds__(KF_TH, 16) kfilter_kernel(const Params P)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    constexpr int VPT = TILE_BYTES / 16;                   // vectors per tile
    constexpr int LOW = (DT == SPEC_F32) ? 0 : 16;          // bf16 keys end at bit 16
    __shared__ KfSmem S;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int V = P.V;
    const int items = P.B * P.rows;
    const size_t NG = (size_t)P.NS * NT;
    allow_next_kernel();
    wait_previous_kernel();  // the partials and the group keys

    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int b = item / P.rows, rsq = item - b * P.rows;
        const float T = __ldg(P.temperature + b);
        const int K = P.top_k ? __ldg(P.top_k + b) : 0;
        const float Pp = P.top_p ? __ldg(P.top_p + b) : 1.0f;
        if (!kf_row(P, T, K, Pp)) {
            // rows with nothing to cut get their record here (as the window
            // kernel writes it); the others are left to the streaming filter
            const bool bad = K < 0 || isnan(Pp) || !(Pp > 0.0f);
            const bool topk = K > 0 && K < V, topp = Pp < 1.0f;
            if (!temperature_valid(T) || T == 0.0f || (!topk && !topp) || bad) {
                if (t == 0) {
                    FiltRec o;
                    o.kappa = 0u;
                    o.iota = INT_MAX;
                    o.zt = 0.0f;
                    o.flags = (temperature_valid(T) && bad) ? FILT_ERR : FILT_OFF;
                    P.filt[item] = o;
                }
            } else if (t == 0) {
                atomicAdd(&P.hdr->n_stream_rows, 1u);
            }
            if (t == 0)
                P.kcount[item] = -1;
            continue;
        }
        const bool topp = Pp < 1.0f;
        const float c = LOG2E / T;
        const float4 *pp = P.part + (size_t)item * P.NSS;
        float m = -INFINITY;
        for (int q = lane; q < P.NSS; q += 32)
            m = fmax_nan(m, __ldcg(pp + q).x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
        FiltRec out;
        out.kappa = 0u;
        out.iota = INT_MAX;
        out.zt = 0.0f;
        out.flags = FILT_OFF;
        int kc = -1;  // kept tokens stored for the kept-set draw (-1: none)
        if (!(isnan(m) || isinf(m))) {  // else the scan reports the row as an error
            const unsigned int *gk = P.gkey + (size_t)item * NG;
            // the group keys, KF_LB loads in flight per thread (from L2 after
            // the first pass).  NG is a multiple of the block, so every lane
            // takes each step.
            auto for_keys = [&](auto fn) {
                for (size_t g0 = 0; g0 < NG; g0 += (size_t)KF_TH * KF_LB) {
                    unsigned int key[KF_LB];
#pragma unroll
                    for (int q = 0; q < KF_LB; ++q) {
                        const size_t g = g0 + (size_t)q * KF_TH + t;
                        key[q] = (g < NG) ? __ldcg(gk + g) : 0u;
                    }
#pragma unroll
                    for (int q = 0; q < KF_LB; ++q)
                        if (g0 + (size_t)q * KF_TH < NG)  // the same in every lane
                            fn(g0 + (size_t)q * KF_TH + t, key[q]);
                }
            };
            // ---- tau: the K-th largest group key, 8 bits per pass
            unsigned int prefix = 0u, pmask = 0u, need = (unsigned int)K;
            for (int shift = 24; shift >= LOW; shift -= 8) {
                for (int i = t; i < 256; i += KF_TH)
                    S.hist[i] = 0u;
                __syncthreads();
                // lanes with the same bin add once, through their leader
                for_keys([&](size_t, unsigned int key) {
                    const bool in = (key & pmask) == prefix;
                    const unsigned int bin = (key >> shift) & 255u;
                    const unsigned int act = __ballot_sync(0xffffffffu, in);
                    if (in) {
                        const unsigned int peers = __match_any_sync(act, bin);
                        if (lane == __ffs(peers) - 1)
                            atomicAdd(&S.hist[bin], (unsigned int)__popc(peers));
                    }
                });
                __syncthreads();
                if (warp == 0) {
                    // lane l holds bins 255 - 8l down to 248 - 8l
                    unsigned int h[8], sum = 0u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        h[j] = S.hist[255 - 8 * lane - j];
                        sum += h[j];
                    }
                    unsigned int incl = sum;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o)
                            incl += y;
                    }
                    const unsigned int excl = incl - sum;
                    const unsigned int hit = __ballot_sync(0xffffffffu, incl >= need);
                    // at least `need` keys match the prefix: some lane hits
                    const int hl = hit ? __ffs(hit) - 1 : 31;
                    if (lane == hl) {
                        unsigned int cum = excl;
                        int sel = 248 - 8 * lane;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if (cum + h[j] >= need) {
                                sel = 255 - 8 * lane - j;
                                break;
                            }
                            cum += h[j];
                        }
                        S.sel = (unsigned int)sel;
                        S.need = need - cum;
                    }
                }
                __syncthreads();
                prefix |= S.sel << shift;
                pmask |= 255u << shift;
                need = S.need;
                __syncthreads();
            }
            const unsigned int tau = prefix;
            // ---- the groups holding a key >= tau, then their tokens >= tau
            if (t == 0) {
                S.ng = 0u;
                S.nc = 0u;
            }
            __syncthreads();
            for_keys([&](size_t g, unsigned int key) {
                const bool sel = key >= tau;
                if (__ballot_sync(0xffffffffu, sel)) {  // most steps select nothing
                    const unsigned int slot = warp_slot(sel, &S.ng, lane);
                    if (sel && slot < (unsigned int)KF_GCAP)
                        S.glist[slot] = (int)g;
                }
            });
            __syncthreads();
            const unsigned int ng = S.ng;
            bool over = ng > (unsigned int)KF_GCAP;
            if (!over) {
                const bool is_target = rsq <= P.k;
                const void *arr = is_target ? P.target : P.draft;
                const size_t row = is_target ? (size_t)b * (P.k + 1) + rsq
                                             : (size_t)b * P.k + (rsq - P.k - 1);
                const int nw = (int)ng * U;
                // the row's vectors are 16-byte aligned in memory when its first
                // element is (the array base is)
                const bool aligned = ((row * (size_t)V) % VEC) == 0;
                const uint4 *rv = reinterpret_cast<const uint4 *>(arr) + (row * (size_t)V) / VEC;
                // KF_GB vectors a thread in flight; every lane takes each step
                for (int w0 = 0; w0 < nw; w0 += KF_TH * KF_GB) {
                    int vv[KF_GB];
                    uint4 raw[KF_GB];
#pragma unroll
                    for (int q = 0; q < KF_GB; ++q) {
                        const int w = w0 + q * KF_TH + t;
                        int v = -1;
                        if (w < nw) {
                            const int g = S.glist[w / U], u = w - (w / U) * U;
                            const int seg = g / NT, gw = (g % NT) / 32, gl = g % 32;
                            v = seg * VPT + 256 * gw + 32 * u + gl;  // the group lane's vector u
                        }
                        vv[q] = v;
                        if (v >= 0 && aligned && (v + 1) * VEC <= V)
                            raw[q] = __ldg(rv + v);
                    }
#pragma unroll
                    for (int q = 0; q < KF_GB; ++q) {
                        if (w0 + q * KF_TH >= nw)
                            break;  // the same in every lane
                        const int v = vv[q];
                        float x[VEC];
                        if (v >= 0 && aligned && (v + 1) * VEC <= V) {
                            L::unpack(raw[q], x);
                        } else {
#pragma unroll
                            for (int j = 0; j < VEC; ++j) {
                                const int e = v * VEC + j;
                                x[j] = (v >= 0 && e < V) ? L::load1(arr, row * (size_t)V + e)
                                                         : -INFINITY;
                            }
                        }
                        // the lane's tokens >= tau, then one range of slots per lane:
                        // a warp scan of the counts and one shared atomic
                        unsigned int mask = 0u;
#pragma unroll
                        for (int j = 0; j < VEC; ++j) {
                            const int e = v * VEC + j;
                            if (v >= 0 && e < V && key_of<DT>(x[j]) >= tau)
                                mask |= 1u << j;
                        }
                        const unsigned int cnt = (unsigned int)__popc(mask);
                        if (__ballot_sync(0xffffffffu, cnt != 0u)) {
                            unsigned int incl = cnt;
#pragma unroll
                            for (int o = 1; o < 32; o <<= 1) {
                                const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
                                if (lane >= o)
                                    incl += y;
                            }
                            unsigned int base = 0u;
                            if (lane == 31)
                                base = atomicAdd(&S.nc, incl);
                            unsigned int slot = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
#pragma unroll
                            for (int j = 0; j < VEC; ++j) {
                                if ((mask >> j) & 1u) {
                                    if (slot < (unsigned int)KF_CAP) {
                                        S.key[slot] = sortkey(key_of<DT>(x[j]), v * VEC + j);
                                        S.mass[slot] = fixmass(x[j], m, c);
                                    }
                                    ++slot;
                                }
                            }
                        }
                    }
                }
                __syncthreads();
                over = S.nc > (unsigned int)KF_CAP;
            }
            if (over) {
                out.flags = FILT_RADIX;
                if (t == 0)
                    atomicAdd(&P.hdr->n_radix_rows, 1u);
            } else {
                // ---- order descending: a token's rank is the number of larger
                // keys (keys are distinct: the index is in them); order[rank]
                // takes the group list's place, no longer needed
                const int n = (int)S.nc;
                int *order = S.glist;
                // the first KF_KMAX in rank order are also stored for the
                // kept-set draw (the kept set is a prefix of them: K <= KF_KMAX)
                unsigned long long *kp = P.kept + (size_t)item * KF_KMAX;
                for (int i = t; i < n; i += KF_TH) {
                    const unsigned long long ki = S.key[i];
                    int r = 0;
                    for (int j = 0; j < n; ++j)
                        r += (S.key[j] > ki) ? 1 : 0;
                    order[r] = i;
                    if (r < KF_KMAX)
                        kp[r] = ki;
                }
                __syncthreads();
                // ---- the cut: the top-k mass, then the top-p end (K <= n)
                const int nk = min(K, n);
                unsigned long long ms = 0ull;
                for (int i = t; i < nk; i += KF_TH)
                    ms += S.mass[order[i]];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    ms += __shfl_xor_sync(0xffffffffu, ms, o);
                if (lane == 0)
                    S.red[warp] = ms;
                __syncthreads();
                unsigned long long ZK = 0ull;
                for (int w = 0; w < KF_TH / 32; ++w)
                    ZK += S.red[w];
                int last = nk - 1;
                unsigned long long Zt = ZK;
                if (topp && warp == 0) {
                    unsigned long long target = (unsigned long long)((double)Pp * (double)ZK);
                    if (target == 0ull)
                        target = 1ull;
                    unsigned long long run = 0ull;
                    int istar = -1;
                    for (int i0 = 0; i0 < nk && istar < 0; i0 += 32) {
                        const int i = i0 + lane;
                        unsigned long long x = (i < nk) ? S.mass[order[i]] : 0ull;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
                            if (lane >= o)
                                x += y;
                        }
                        const unsigned long long inc = run + x;
                        const unsigned int hit = __ballot_sync(0xffffffffu, i < nk && inc >= target);
                        if (hit) {
                            const int hl = __ffs(hit) - 1;
                            istar = i0 + hl;
                            run = __shfl_sync(0xffffffffu, inc, hl);
                        } else {
                            run = __shfl_sync(0xffffffffu, inc, 31);
                        }
                    }
                    if (istar < 0)
                        istar = nk - 1;  // rounding: all of them
                    last = istar;
                    Zt = run;
                }
                const unsigned long long e = S.key[order[last]];
                kc = last + 1;  // thread 0's is the one stored
                out.kappa = (unsigned int)(e >> 32);
                out.iota = (int)(0xffffffffu - (unsigned int)(e & 0xffffffffu));
                out.zt = (float)((double)Zt * (1.0 / 1099511627776.0));
                out.flags = FILT_ON;
            }
        }
        if (t == 0) {
            P.filt[item] = out;
            P.kcount[item] = kc;
        }
        __syncthreads();  // the row's shared state is free again
    }
}

// ------------------------------------ top-k / top-p: the one-pass window kernel
//
// The common case of the filter, warp-specialized like the statistics kernel:
// a producer warp deals rows (the header counter) and streams each filtered
// row through a ring of 16 KB bulk copies without stopping between rows;
// eight consumer warps each take a contiguous 2 KB of every tile into
// registers, free the slot, and gather the row's window tokens (the
// adaptive window of filter_kernel, described there).  Each warp narrows its
// own copy of the window from the shared histogram: counts only grow, so the
// bin it reads as the cut's is never below the row's final one, and every
// token of the bins through the final cut is gathered by every warp.  Block
// work (the cut from the sorted window) is done once per row between
// barriers of the consumer warps, each a bounded mbarrier wait.  A row whose
// buffer overflowed, or whose window ended short of the cut, is recorded
// FILT_RADIX and finished by filter_kernel.
constexpr int WCW = 8;                            // consumer warps
constexpr int WPW = WCW;                          // the producer's warp
constexpr int WTH = (WCW + 1) * 32;
constexpr int WSLOTS = 4;
constexpr int WVPL = FTILE / (16 * 32 * WCW);     // 16-byte vectors per lane per tile
static_assert(WVPL * 16 * 32 * WCW == FTILE, "a window tile splits evenly over the consumers");
static_assert(WCW * 32 == FTH, "the consumers are the filter's thread count");
enum { WKIND_ROW = 1, WKIND_END = 2 };

struct WTile {
    int kind;
    int item;          // the row (sequence * rows + row in sequence)
    int e0, e1;        // elements of the row in the slot
    int phase0, ncopied;
    int first, last;   // first / last tile of the row
};

struct WSmem {
    uint8_t ring[WSLOTS][FSLOT_BYTES];
    unsigned long long full[WSLOTS];
    unsigned long long empty[WSLOTS];
    WTile tile[WSLOTS];
    unsigned long long ckey[FCAP], cmass[FCAP];  // the window's tokens
    unsigned long long rkey[FCAP], rmass[FCAP];  // compaction / sort output
    unsigned int fh_cnt[WBINS];
    unsigned long long fh_mass[WBINS];
    unsigned int ncand;
    int overflow;
    unsigned int wcnt[WCW];
    int wnb;
    unsigned int wcum;
    int sel;
    unsigned long long acc;
    unsigned long long cbar;  // the consumers' barrier (every consumer thread arrives)
    int abort_flag;
};
constexpr size_t WFILT_SMEM = sizeof(WSmem);

template <int DT>
__global__ void __launch_bounds__(WTH, 2) wfilter_kernel(const Params P)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    constexpr int TE = FTILE / L::ES;  // elements per tile
    extern __shared__ __align__(16) uint8_t wsm_raw[];
    WSmem &S = *reinterpret_cast<WSmem *>(wsm_raw);
    volatile int *abort_flag = &S.abort_flag;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int V = P.V;
    const int items = P.B * P.rows;
    const int ntiles = (V + TE - 1) / TE;
    if (t == 0) {
        for (int q = 0; q < WSLOTS; ++q) {
            mbar_init(&S.full[q], 1);
            mbar_init(&S.empty[q], WCW);
        }
        mbar_init(&S.cbar, WCW * 32);
        S.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    allow_next_kernel();
    wait_previous_kernel();  // the partials and the zeroed row counter
    if (P.gkey && __ldcg(&P.hdr->n_stream_rows) == 0u)
        return;  // the group-maximum cut took every row that needed a cut

    if (warp == WPW) {
        // ---------------------------------------------------------- producer
        if (lane != 0)
            return;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0u, issued_phase = 0u;
        bool ok = true;
        for (int item = blockIdx.x; item < items && ok;
             item = (int)gridDim.x + (int)atomicAdd(&P.hdr->next_item, 1u)) {
            const int b = item / P.rows, rsq = item - b * P.rows;
            const float T = __ldg(P.temperature + b);
            const int K = P.top_k ? __ldg(P.top_k + b) : 0;
            const float Pp = P.top_p ? __ldg(P.top_p + b) : 1.0f;
            const bool topk = K > 0 && K < V;
            const bool topp = Pp < 1.0f;
            const bool bad = K < 0 || isnan(Pp) || !(Pp > 0.0f);
            if (kf_row(P, T, K, Pp))
                continue;  // cut from the group maxima (kfilter_kernel)
            if (!temperature_valid(T) || T == 0.0f || (!topk && !topp) || bad) {
                FiltRec out;
                out.kappa = 0u;
                out.iota = INT_MAX;
                out.zt = 0.0f;
                // bad filter parameters fail the sequence, greedy too; greedy,
                // invalid and unfiltered rows keep everything
                out.flags = (temperature_valid(T) && bad) ? FILT_ERR : FILT_OFF;
                P.filt[item] = out;
                continue;
            }
            const bool is_target = rsq <= P.k;
            const uint8_t *arr = reinterpret_cast<const uint8_t *>(is_target ? P.target : P.draft);
            const size_t row = is_target ? (size_t)b * (P.k + 1) + rsq
                                         : (size_t)b * P.k + (rsq - P.k - 1);
            const unsigned long long arr_bytes = is_target ? P.target_bytes : P.draft_bytes;
            for (int i = 0; i < ntiles; ++i) {
                if (*abort_flag || !mbar_wait(&S.empty[stage], phase ^ 1u)) {
                    ok = false;
                    break;
                }
                const int e0 = i * TE, e1 = min(V, e0 + TE);
                const unsigned long long start = ((unsigned long long)row * V + e0) * L::ES;
                const unsigned long long end = ((unsigned long long)row * V + e1) * L::ES;
                const unsigned long long a0 = start & ~15ull;
                unsigned long long a1 = (end + 15) & ~15ull;
                if (a1 > (arr_bytes & ~15ull))
                    a1 = arr_bytes & ~15ull;
                const uint32_t bytes = (a1 > a0) ? (uint32_t)(a1 - a0) : 0u;
                WTile &ti = S.tile[stage];
                ti.kind = WKIND_ROW;
                ti.item = item;
                ti.e0 = e0;
                ti.e1 = e1;
                ti.phase0 = (int)(start - a0);
                ti.ncopied = (int)bytes;
                ti.first = (i == 0) ? 1 : 0;
                ti.last = (i == ntiles - 1) ? 1 : 0;
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                if (bytes) {
                    mbar_arrive_expect_tx(&S.full[stage], bytes);
                    bulk_copy_g2s(S.ring[stage], arr + a0, bytes, &S.full[stage]);
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                } else {
                    mbar_arrive(&S.full[stage]);
                }
                if (++stage == WSLOTS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (ok) {  // the end marker
            if (!*abort_flag && mbar_wait(&S.empty[stage], phase ^ 1u)) {
                S.tile[stage].kind = WKIND_END;
                mbar_arrive(&S.full[stage]);
            } else {
                ok = false;
            }
        }
        if (!ok) {
            atomicExch(&P.hdr->status, SPEC_DEV_WAIT_TIMEOUT);
            *abort_flag = 1;
            for (int q = 0; q < WSLOTS; ++q)  // the copies in flight land first (bounded)
                if ((issued >> q) & 1u)
                    (void)mbar_wait(&S.full[q], (issued_phase >> q) & 1u);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int vwarp = warp * 32 * WVPL;  // this warp's first vector of a tile
    int stage = 0;
    uint32_t phase = 0;
    // the current row (the same in every warp)
    int item = -1;
    float m = 0.0f, c = 0.0f, Pp = 1.0f;
    int K = 0, nbw0 = -1, nbw = -1;  // nbw: this warp's window (bins 0..nbw)
    bool topk = false, topp = false, need_mass = false, row_bad = false;
    unsigned long long Zrow = 0ull, target0 = 0ull;
    unsigned int kmin = 1u, last_nc = 0u;
    // The consumers' barrier is an mbarrier every consumer thread arrives at
    // and waits on with the bounded wait, so a warp that gave up on a copy
    // makes the others give up too instead of stopping them for good.  A
    // thread that gave up (dead) skips the rest; the verdict is per warp.
    uint32_t cphase = 0u;
    bool dead = false;
    auto cbar = [&]() {
        if (dead)
            return;
        mbar_arrive(&S.cbar);
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&S.cbar, cphase));
        cphase ^= 1u;
        if (!ok) {
            dead = true;
            if (lane == 0) {
                atomicExch(&P.hdr->status, SPEC_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
            }
        }
    };
    // exclusive prefix over the consumer threads (index order = thread order)
    auto block_scan = [&](unsigned int x, unsigned int &total) -> unsigned int {
        unsigned int incl = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        if (lane == 31)
            S.wcnt[warp] = incl;
        cbar();
        unsigned int wbase = 0, tot = 0;
        for (int w = 0; w < WCW; ++w) {
            const unsigned int v = S.wcnt[w];
            if (w < warp)
                wbase += v;
            tot += v;
        }
        cbar();
        total = tot;
        return wbase + incl - x;
    };

    auto wbin = [&](float x) {
        const float dd = (m - x) * c;
        return (dd < (float)(WBINS / 2)) ? (int)(dd * 2.0f) : WBINS;
    };
    auto val_of_key = [&](unsigned int key) {
        unsigned int bits = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
        if (DT == SPEC_BF16)
            bits &= 0xffff0000u;
        return __uint_as_float(bits);
    };
    // The window's lower edge: the smallest float x with wbin(x) <= lim.
    // wbin is monotone in x (each rounding step is), so a token is inside the
    // window iff x >= edge, one compare instead of the bin computation.
    // Found by bisection on the order keys between a value one bit outside
    // the window and the row maximum (inside); each step evaluates wbin, the
    // same expression the bins are counted with.
    auto edge_of = [&](int lim) -> float {
        auto fkey = [](float x) { return okey(__float_as_uint(x)); };
        auto kval = [](unsigned int k) {
            return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
        };
        unsigned int lo = fkey(m - ((float)lim * 0.5f + 2.0f) / c);  // wbin(lo) > lim
        unsigned int hi = fkey(m);                                      // wbin(m) = 0 <= lim
        while (hi - lo > 1u) {
            const unsigned int mid = lo + (hi - lo) / 2u;
            if (wbin(kval(mid)) <= lim)
                hi = mid;
            else
                lo = mid;
        }
        return kval(hi);
    };
    float xs = 0.0f, xs0 = 0.0f;  // the edges of this warp's window and of the first
    // this warp's reading of the first bin (<= lim) whose counts (masses)
    // reach the cut, and the count through it; -1 if none
    auto warp_bk = [&](int lim, unsigned int &cum_out) -> int {
        volatile unsigned int *fc = S.fh_cnt;
        volatile unsigned long long *fm = S.fh_mass;
        const int b0 = 2 * lane, b1 = b0 + 1;
        const unsigned int c0 = (b0 <= lim) ? fc[b0] : 0u;
        const unsigned int c1 = (b1 <= lim) ? fc[b1] : 0u;
        const unsigned long long m0 = (need_mass && b0 <= lim) ? fm[b0] : 0ull;
        const unsigned long long m1 = (need_mass && b1 <= lim) ? fm[b1] : 0ull;
        unsigned int ci = c0 + c1;
        unsigned long long mi = m0 + m1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned int y = __shfl_up_sync(0xffffffffu, ci, o);
            const unsigned long long ym = __shfl_up_sync(0xffffffffu, mi, o);
            if (lane >= o) {
                ci += y;
                mi += ym;
            }
        }
        const unsigned int ce0 = ci - c1;
        const unsigned long long me0 = mi - m1;
        auto hits = [&](unsigned int cc, unsigned long long mm) {
            return topk ? cc >= (unsigned int)K : mm >= target0;
        };
        const bool h0 = b0 <= lim && hits(ce0, me0);
        const bool h1 = b1 <= lim && hits(ci, mi);
        const unsigned int hb = __ballot_sync(0xffffffffu, h0 || h1);
        if (!hb) {
            cum_out = 0u;
            return -1;
        }
        const int L0 = __ffs(hb) - 1;
        const bool first0 = __shfl_sync(0xffffffffu, h0, L0);
        cum_out = __shfl_sync(0xffffffffu, first0 ? ce0 : ci, L0);
        return first0 ? 2 * L0 : 2 * L0 + 1;
    };

    for (;;) {
        if (dead)
            break;
        int ok = 1;
        if (lane == 0)
            ok = mbar_wait(&S.full[stage], phase) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0) {
                atomicExch(&P.hdr->status, SPEC_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
            }
            break;
        }
        (void)mbar_try_wait(&S.full[stage], phase);  // acquire the landed bytes
        const WTile ti = S.tile[stage];
        if (ti.kind == WKIND_END)
            break;
        if (ti.first) {
            // a new row: its parameters (each warp computes the same values)
            item = ti.item;
            const int b = item / P.rows, rsq = item - b * P.rows;
            const float T = __ldg(P.temperature + b);
            K = P.top_k ? __ldg(P.top_k + b) : 0;
            Pp = P.top_p ? __ldg(P.top_p + b) : 1.0f;
            topk = K > 0 && K < V;
            topp = Pp < 1.0f;
            need_mass = !topk;
            c = LOG2E / T;
            const float4 *pp = P.part + ((size_t)b * P.rows + rsq) * P.NSS;
            float mm = -INFINITY;
            for (int q = lane; q < P.NSS; q += 32)
                mm = fmax_nan(mm, __ldcg(pp + q).x);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                mm = fmax_nan(mm, __shfl_xor_sync(0xffffffffu, mm, o));
            float z = 0.0f;
            for (int q = lane; q < P.NSS; q += 32) {
                const float4 pv = __ldcg(pp + q);
                z += rescale(pv.y, pv.x, mm, c);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                z += __shfl_xor_sync(0xffffffffu, z, o);
            m = mm;
            row_bad = isnan(m) || isinf(m);  // the scan reports the row as an error
            Zrow = (unsigned long long)((double)z * 1099511627776.0);
            target0 = topk ? 0ull : (unsigned long long)((double)Pp * (double)Zrow);
            const float zrow = (float)((double)Zrow * (1.0 / 1099511627776.0));
            const int Dg = (int)floorf(log2f((float)FCAP / (fmaxf(zrow, 1.0f) * 1.01f))) + 8;
            nbw0 = nbw = row_bad ? -1 : 2 * min(WBINS / 2, max(1, Dg)) - 1;
            if (!row_bad)
                xs0 = xs = edge_of(nbw0);
            kmin = topk ? (unsigned int)K : 1u;
            last_nc = 0u;
            if (t == 0) {
                S.ncand = 0u;
                S.overflow = 0;
            }
            if (t < WBINS) {
                S.fh_cnt[t] = 0u;
                S.fh_mass[t] = 0ull;
            }
            cbar();  // the previous row's cut is done; the window state is reset
        }
        // this warp's 2 KB of the tile into registers, then the slot is free
        const Seg g = make_seg<DT>(S.ring[stage], nullptr, 0, V, ti.e0, ti.e1, ti.phase0,
                                   ti.ncopied);
        const int vt0 = ti.e0 / VEC;
        uint4 raw[WVPL];
        if (g.fast && ti.e1 - ti.e0 == TE) {
#pragma unroll
            for (int u = 0; u < WVPL; ++u)
                raw[u] = ld_shared_v4(S.ring[stage] + (size_t)(vwarp + lane + 32 * u) * 16);
        } else {
            // the row's array is only read for bytes the copy left out (none
            // when the row is 16-byte aligned)
            const bool is_t = (item % P.rows) <= P.k;
            const int bq = item / P.rows, rq = item - bq * P.rows;
            const size_t rrow = is_t ? (size_t)bq * (P.k + 1) + rq : (size_t)bq * P.k + (rq - P.k - 1);
            const Seg g2 = make_seg<DT>(S.ring[stage], is_t ? P.target : P.draft, rrow, V, ti.e0,
                                        ti.e1, ti.phase0, ti.ncopied);
#pragma unroll
            for (int u = 0; u < WVPL; ++u)
                raw[u] = seg_vec<DT>(g2, vt0 + vwarp + lane + 32 * u);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&S.empty[stage]);
        if (++stage == WSLOTS) {
            stage = 0;
            phase ^= 1u;
        }

        // ---- the window gather (per lane marks, one slot reservation per warp).
        // The vectors rotate through r0..r3 so that each loop below is one
        // short body, not unrolled: the hot loop stays small enough for the
        // instruction cache (four rotations bring them back in order).
        // A row's first tile goes through twice: first its tokens inside the
        // first window are only counted, and every warp narrows to the bin
        // where those counts reach the cut (the counts of the whole row can
        // only be larger, so the row's cut bin is not past it); then the
        // tile's tokens inside that window are stored.  A wide first window
        // on a flat row therefore does not flood the buffer.
        // Decisions that guard warp collectives are taken from lane 0's read
        // of shared state and broadcast: lanes reading it at different times
        // (another warp may change it in between) must not split the warp.
        int ovf = 0;
        if (lane == 0)
            ovf = *(volatile int *)&S.overflow;
        ovf = __shfl_sync(0xffffffffu, ovf, 0);
        if (!row_bad && !ovf) {
            const int npass = ti.first ? 2 : 1;
#pragma unroll 1
            for (int pass = 0; pass < npass; ++pass) {
                const bool count_only = ti.first && pass == 0;
                const bool count = !ti.first || pass == 0;
                const float xe = count_only ? xs0 : xs;  // the window: x >= xe
                uint4 r0 = raw[0], r1 = raw[1], r2 = raw[2], r3 = raw[3];
                static_assert(WVPL == 4 && VEC <= 8, "four vectors of at most 8 tokens per lane");
                uint32_t tball = 0u;  // 8 bits per vector: the tokens in the window
                unsigned int cnt = 0u;
#pragma unroll
                for (int u = 0; u < WVPL; ++u) {
                    uint32_t tb = 0u;
                    if (L::vmax(raw[u]) >= xe) {  // else no token of the vector is in
                        float x[VEC];
                        L::unpack(raw[u], x);
#pragma unroll
                        for (int j = 0; j < VEC; ++j)
                            tb |= (x[j] >= xe) ? (1u << j) : 0u;
                        const int idx0 = (vt0 + vwarp + lane + 32 * u) * VEC;
                        if (idx0 + VEC > V)  // the row's end
                            tb &= (V > idx0) ? ((1u << (V - idx0)) - 1u) : 0u;
                    }
                    tball |= tb << (8 * u);
                    cnt += (unsigned int)__popc(tb);
                }
                unsigned int pos = 0u;
                bool any = true;
                if (!count_only) {
                    unsigned int incl = cnt;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o)
                            incl += y;
                    }
                    const unsigned int wtot = __shfl_sync(0xffffffffu, incl, 31);
                    any = wtot != 0u;
                    if (any) {
                        unsigned int base = 0u;
                        if (lane == 31)
                            base = atomicAdd(&S.ncand, wtot);
                        base = __shfl_sync(0xffffffffu, base, 31);
                        if (base + wtot > (unsigned int)FCAP && lane == 0)
                            S.overflow = 1;  // tokens not stored: the radix search finishes the row
                        pos = base + incl - cnt;
                    }
                }
                if (any && tball) {
#pragma unroll 1
                    for (int u = 0; u < WVPL; ++u) {
                        const uint32_t tb = (tball >> (8 * u)) & 0xffu;
                        if (tb) {
                            float x[VEC];
                            L::unpack(r0, x);
#pragma unroll
                            for (int j = 0; j < VEC; ++j) {
                                if ((tb >> j) & 1u) {
                                    const bool keep = !count_only && pos < (unsigned int)FCAP;
                                    const unsigned long long e =
                                        (keep || (count && need_mass)) ? fixmass(x[j], m, c) : 0ull;
                                    if (count) {
                                        const int wb = wbin(x[j]);
                                        atomicAdd(&S.fh_cnt[wb], 1u);
                                        if (need_mass)
                                            atomicAdd(&S.fh_mass[wb], e);
                                    }
                                    if (keep) {
                                        const int idx = (vt0 + vwarp + lane + 32 * u) * VEC + j;
                                        S.ckey[pos] = sortkey(key_of<DT>(x[j]), idx);
                                        S.cmass[pos] = e;
                                    }
                                    ++pos;
                                }
                            }
                        }
                        const uint4 rt = r0;
                        r0 = r1;
                        r1 = r2;
                        r2 = r3;
                        r3 = rt;
                    }
                }
                if (count_only) {
                    cbar();  // every warp's counts of the first tile are in
                    unsigned int cum0;
                    const int bk0 = warp_bk(nbw0, cum0);
                    if (bk0 >= 0 && bk0 < nbw) {
                        nbw = bk0;
                        xs = edge_of(nbw);
                    }
                }
            }
            // narrow this warp's window once the gathered count has doubled
            unsigned int nc = 0u;
            if (lane == 0)
                nc = *(volatile unsigned int *)&S.ncand;
            nc = __shfl_sync(0xffffffffu, nc, 0);  // (the same decision in every lane)
            if (nc >= kmin && nc >= 2u * last_nc) {
                last_nc = nc;
                unsigned int cum;
                const int bk = warp_bk(nbw, cum);
                if (bk >= 0 && bk < nbw) {
                    nbw = bk;
                    xs = edge_of(nbw);
                }
            }
        }
        if (!ti.last)
            continue;

        // ---- end of the row: the cut from the sorted window (all consumers)
        cbar();  // every warp's tokens of the row are in
        if (dead)
            break;
        FiltRec out;
        out.kappa = 0u;
        out.iota = INT_MAX;
        out.zt = 0.0f;
        out.flags = FILT_OFF;
        if (!row_bad) {
            unsigned int ncut = 0u;
            const int bk = S.overflow ? -1 : warp_bk(nbw0, ncut);  // the same in every warp
            if (bk < 0) {
                out.flags = FILT_RADIX;
            } else {
                int n = (int)S.ncand;
                const unsigned long long *sk = S.ckey, *sm = S.cmass;
                if ((int)ncut < n) {
                    // only the bins through the cut's (wider warps gathered more)
                    constexpr int PER = FCAP / FTH;
                    bool kp[PER];
                    unsigned int cnt = 0u;
#pragma unroll
                    for (int q = 0; q < PER; ++q) {
                        const int i = t * PER + q;
                        kp[q] = i < n && wbin(val_of_key((unsigned int)(S.ckey[i] >> 32))) <= bk;
                        cnt += kp[q] ? 1u : 0u;
                    }
                    unsigned int total;
                    unsigned int o = block_scan(cnt, total);
#pragma unroll
                    for (int q = 0; q < PER; ++q) {
                        const int i = t * PER + q;
                        if (kp[q]) {
                            S.rkey[o] = S.ckey[i];
                            S.rmass[o] = S.cmass[i];
                            ++o;
                        }
                    }
                    cbar();
                    n = (int)total;
                    sk = S.rkey;
                    sm = S.rmass;
                }
                // sort descending by (key, -index): the ranking
                unsigned long long *dk, *dm;
                if (n <= FCAP / 2) {
                    // rank placement (keys are unique) into the other buffer
                    dk = (sk == S.ckey) ? S.rkey : S.ckey;
                    dm = (sk == S.ckey) ? S.rmass : S.cmass;
                    constexpr int PER2 = FCAP / 2 / FTH;
                    unsigned long long mine[PER2], mm[PER2];
                    int rk[PER2];
#pragma unroll
                    for (int q = 0; q < PER2; ++q) {
                        const int i = t + q * FTH;
                        mine[q] = (i < n) ? sk[i] : 0ull;
                        mm[q] = (i < n) ? sm[i] : 0ull;
                        rk[q] = 0;
                    }
                    for (int jj = 0; jj < n; ++jj) {
                        const unsigned long long kj = sk[jj];
#pragma unroll
                        for (int q = 0; q < PER2; ++q)
                            rk[q] += (kj > mine[q]) ? 1 : 0;
                    }
#pragma unroll
                    for (int q = 0; q < PER2; ++q) {
                        const int i = t + q * FTH;
                        if (i < n) {
                            dk[rk[q]] = mine[q];
                            dm[rk[q]] = mm[q];
                        }
                    }
                    cbar();
                } else {
                    // bitonic, in place, padded to a power of two
                    dk = const_cast<unsigned long long *>(sk);
                    dm = const_cast<unsigned long long *>(sm);
                    int p2 = 1;
                    while (p2 < n)
                        p2 <<= 1;
                    for (int i = n + t; i < p2; i += FTH) {
                        dk[i] = 0ull;
                        dm[i] = 0ull;
                    }
                    cbar();
                    for (int kk = 2; kk <= p2; kk <<= 1) {
                        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                            for (int i = t; i < p2; i += FTH) {
                                const int ixj = i ^ jj;
                                if (ixj > i) {
                                    const unsigned long long a = dk[i], bq = dk[ixj];
                                    const bool desc = (i & kk) == 0;
                                    if (desc ? (a < bq) : (a > bq)) {
                                        dk[i] = bq;
                                        dk[ixj] = a;
                                        const unsigned long long ma = dm[i];
                                        dm[i] = dm[ixj];
                                        dm[ixj] = ma;
                                    }
                                }
                            }
                            cbar();
                        }
                    }
                }
                // the cuts, read off the sorted list by every warp alike
                // (K <= n: the counts through the cut's bin reached K)
                const int nk = min(topk ? K : n, n);
                unsigned long long ZK;
                {
                    unsigned long long ms = 0ull;
                    for (int i = lane; i < nk; i += 32)
                        ms += dm[i];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        ms += __shfl_xor_sync(0xffffffffu, ms, o);
                    ZK = topk ? ms : Zrow;
                }
                int last = nk - 1;
                unsigned long long Zt = ZK;
                if (topp) {
                    unsigned long long target = (unsigned long long)((double)Pp * (double)ZK);
                    if (target == 0ull)
                        target = 1ull;
                    unsigned long long run = 0ull;
                    int istar = -1;
                    for (int i0 = 0; i0 < nk && istar < 0; i0 += 32) {
                        const int i = i0 + lane;
                        unsigned long long x = (i < nk) ? dm[i] : 0ull;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
                            if (lane >= o)
                                x += y;
                        }
                        const unsigned long long inc = run + x;
                        const unsigned int hit = __ballot_sync(0xffffffffu, i < nk && inc >= target);
                        if (hit) {
                            const int hl = __ffs(hit) - 1;
                            istar = i0 + hl;
                            run = __shfl_sync(0xffffffffu, inc, hl);
                        } else {
                            run = __shfl_sync(0xffffffffu, inc, 31);
                        }
                    }
                    if (istar < 0)
                        istar = nk - 1;  // rounding: all of them
                    last = istar;
                    Zt = run;
                }
                const unsigned long long e = dk[last];
                out.kappa = (unsigned int)(e >> 32);
                out.iota = (int)(0xffffffffu - (unsigned int)(e & 0xffffffffu));
                out.zt = (float)((double)Zt * (1.0 / 1099511627776.0));
                out.flags = FILT_ON;
            }
        }
        if (t == 0) {
            P.filt[item] = out;
            if (out.flags == FILT_RADIX)
                atomicAdd(&P.hdr->n_radix_rows, 1u);
        }
        cbar();  // every warp is done with the row's shared state
    }
}

// -------------------------------------------------------------- accept scan

template <int DT, bool FILT>
__global__ void __launch_bounds__(SCAN_WARPS * 32) scan_kernel(const Params P)
{
    using L = Lg<DT>;
    __shared__ float rm[SCAN_WARPS][MAX_ROWS], rZ[SCAN_WARPS][MAX_ROWS];
    __shared__ int rarg[SCAN_WARPS][MAX_ROWS], rbad[SCAN_WARPS][MAX_ROWS];
    __shared__ unsigned int rkap[FILT ? SCAN_WARPS : 1][FILT ? MAX_ROWS : 1];
    __shared__ int riota[FILT ? SCAN_WARPS : 1][FILT ? MAX_ROWS : 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * SCAN_WARPS + warp;
    if (b >= P.B)
        return;
    const int k = P.k, V = P.V;
    // every load that depends on no other goes out first: the temperature, the
    // tokens and uniforms, and the partials of every row (whether or not the
    // sequence's mode needs them)
    const float T = __ldg(P.temperature + b);
    const int g = (lane < k) ? __ldg(P.tokens + (size_t)b * k + lane) : 0;
    const float ua = (lane < k) ? __ldg(P.u_accept + (size_t)b * k + lane) : 0.0f;
    const float ur = __ldg(P.u_resample + b);
    allow_next_kernel();
    wait_previous_kernel();  // the partials come from the statistics kernel
    constexpr int PRE = 8;
    float4 pre[PRE];
    if (lane < P.rows) {
        const float4 *pp = P.part + ((size_t)b * P.rows + lane) * P.NSS;
#pragma unroll
        for (int q = 0; q < PRE; ++q)
            if (q < P.NSS)
                pre[q] = __ldcg(pp + q);
    }
    const bool tvalid = temperature_valid(T);
    const bool greedy = tvalid && T == 0.0f;
    const float c = (tvalid && !greedy) ? LOG2E / T : 0.0f;

    // 1. fold each row's super-tile partials left to right (one lane per row)
    const int nrows = tvalid ? (greedy ? k + 1 : P.rows) : 0;
    for (int r = lane; r < nrows; r += 32) {
        float m = -INFINITY, s = 0.0f;
        int idx = INT_MAX;
        auto fold = [&](const float4 &pv) {
            const float pm = pv.x, ps = pv.y;
            const int pi = __float_as_int(pv.z);
            const float mn = fmax_nan(m, pm);
            if (!greedy)
                s = rescale(s, m, mn, c) + rescale(ps, pm, mn, c);
            idx = (m == mn && pm == mn) ? min(idx, pi) : (pm == mn ? pi : idx);
            m = mn;
        };
        const float4 *pp = P.part + ((size_t)b * P.rows + r) * P.NSS;
        int q = 0;
        if (r == lane) {
#pragma unroll
            for (int qq = 0; qq < PRE; ++qq)
                if (qq < P.NSS)
                    fold(pre[qq]);
            q = PRE;
        }
        for (; q < P.NSS; ++q)
            fold(__ldcg(pp + q));
        rm[warp][r] = m;
        rZ[warp][r] = s;
        rarg[warp][r] = idx;
        rbad[warp][r] = (isnan(m) || isinf(m)) ? 1 : 0;  // NaN, +inf, or all -inf
    }
    // filtered calls: the kept set of each row (the whole row when unfiltered)
    bool ferr = false, fon = false;
    if constexpr (FILT) {
        for (int r = lane; r < P.rows; r += 32) {
            const FiltRec f = P.filt[(size_t)b * P.rows + r];
            rkap[warp][r] = f.kappa;
            riota[warp][r] = f.iota;
            if (f.flags == FILT_ON && r < nrows)
                rZ[warp][r] = f.zt;
            ferr |= f.flags == FILT_ERR;
            fon |= f.flags == FILT_ON;
        }
        ferr = __any_sync(0xffffffffu, ferr);
        fon = __any_sync(0xffffffffu, fon);
    }
    __syncwarp();

    // 2. accept scan: lane i tests position i
    bool err = !tvalid || ferr;
    bool fail = false, qzero = false;
    if (!err) {
        if (lane < k && (g < 0 || g >= V))
            err = true;
        for (int r = lane; r < nrows; r += 32)
            if (rbad[warp][r])
                err = true;
        err = __any_sync(0xffffffffu, err);
    }
    int j = k, token = -1;
    if (!err) {
        if (greedy) {
            fail = (lane < k) && (g != rarg[warp][lane]);
        } else if (lane < k) {
            const size_t rt = (size_t)b * (k + 1) + lane, rd = (size_t)b * k + lane;
            const float lt = L::load1(P.target, rt * V + g);
            const float ld = L::load1(P.draft, rd * V + g);
            const float mt = rm[warp][lane], zt = rZ[warp][lane];
            const float md = rm[warp][k + 1 + lane], zd = rZ[warp][k + 1 + lane];
            bool in_t = true, in_d = true;  // g in the target's / draft's kept set
            if constexpr (FILT) {
                const unsigned int kt_ = key_of<DT>(lt), kd_ = key_of<DT>(ld);
                in_t = kt_ > rkap[warp][lane] || (kt_ == rkap[warp][lane] && g <= riota[warp][lane]);
                in_d = kd_ > rkap[warp][k + 1 + lane] ||
                       (kd_ == rkap[warp][k + 1 + lane] && g <= riota[warp][k + 1 + lane]);
            }
            qzero = (ld == -INFINITY) || !in_d;
            const float dt = lt - mt, dd = ld - md;
            const float x = (dt - dd) * c;
            const float ratio = in_t ? ((x == 0.0f) ? 1.0f : ex2(x)) * (zd / zt) : 0.0f;
            fail = qzero || !((ratio >= 1.0f) || (ua < ratio));
            if (P.out_probs) {
                P.out_probs[((size_t)b * k + lane) * 2 + 0] = in_t ? ex2(dt * c) / zt : 0.0f;
                P.out_probs[((size_t)b * k + lane) * 2 + 1] = in_d ? ex2(dd * c) / zd : 0.0f;
            }
        }
        const unsigned fm = __ballot_sync(0xffffffffu, fail);
        j = fm ? (__ffs(fm) - 1) : k;
        if (!greedy) {
            const unsigned qm = __ballot_sync(0xffffffffu, qzero);
            if (j < k && ((qm >> j) & 1u))
                err = true;
        } else {
            token = rarg[warp][j];
        }
    }
    if (P.out_probs && (err || greedy) && lane < k) {
        P.out_probs[((size_t)b * k + lane) * 2 + 0] = __int_as_float(0x7fc00000);
        P.out_probs[((size_t)b * k + lane) * 2 + 1] = __int_as_float(0x7fc00000);
    }
    JobRec J;
    J.b = b;
    J.j = j;
    J.filt = 0;
    J.pad0 = J.pad1 = 0;
    J.kt = J.kd = 0u;
    J.it = J.id = INT_MAX;
    if (err || greedy) {
        for (int i = lane; i <= k; i += 32) {
            int o = -1;
            if (!err)
                o = (i < j) ? __ldg(P.tokens + (size_t)b * k + i) : (i == j ? token : -1);
            P.out_tokens[(size_t)b * (k + 1) + i] = o;
        }
        if (lane == 0)
            P.out_num_accepted[b] = err ? -1 : j;
        J.mode = DRAW_NONE;
        J.c = J.u = J.mt = J.rzt = J.md = J.rzd = 0.0f;
        J.t_row = J.d_row = 0;
    } else {
        // the residual at the rejected position, or the bonus row
        J.c = c;
        J.u = ur;
        J.t_row = (long long)b * (k + 1) + j;
        J.mt = rm[warp][j];
        J.rzt = 1.0f / rZ[warp][j];
        if (j < k) {
            J.mode = DRAW_RESIDUAL;
            J.d_row = (long long)b * k + j;
            J.md = rm[warp][k + 1 + j];
            J.rzd = 1.0f / rZ[warp][k + 1 + j];
        } else {
            J.mode = DRAW_TARGET;
            J.d_row = J.t_row;
            J.md = J.mt;
            J.rzd = J.rzt;
        }
        if constexpr (FILT) {
            if (fon) {
                J.filt = 1;
                J.kt = rkap[warp][j];
                J.it = riota[warp][j];
                J.kd = (j < k) ? rkap[warp][k + 1 + j] : J.kt;
                J.id = (j < k) ? riota[warp][k + 1 + j] : J.it;
                // top-k rows with group maxima: drawn from the kept sets alone
                const int K = P.top_k ? __ldg(P.top_k + b) : 0;
                J.pad0 = (P.gkey && K > 0 && K < V && K <= KF_KMAX) ? 1 : 0;
            }
            // the draws the streaming draw kernel still has to serve
            if (lane == 0 && !J.pad0 && (J.mode == DRAW_RESIDUAL || J.filt))
                atomicAdd(&P.hdr->n_stream_draws, 1u);
        }
    }
    if (lane < JOB_VECS)
        reinterpret_cast<uint4 *>(P.jobs + b)[lane] = reinterpret_cast<const uint4 *>(&J)[lane];
}

// ------------------------------------------------------------ draw weights
//
// w(x) = max(0, p(x) - q(x)) (residual) or the unnormalised target weight
// 2^((t(x)-m)*c) (bonus, or the rounding-only fallback).  -inf padding gives 0.

template <int DT, bool FILT>
__device__ __forceinline__ void draw_weights(const JobRec &J, int mode, const uint4 &rt,
                                             const uint4 &rd, float (&w)[Lg<DT>::VEC], int e0)
{
    using L = Lg<DT>;
    float xt[L::VEC];
    L::unpack(rt, xt);
    // top-k / top-p: tokens outside a row's kept set weigh nothing in it
    auto kept = [&](float x, int j, unsigned int kap, int iota) {
        if constexpr (!FILT) {
            return true;
        } else {
            if (!J.filt)
                return true;
            const unsigned int key = key_of<DT>(x);
            return key > kap || (key == kap && e0 + j <= iota);
        }
    };
    if (mode == DRAW_RESIDUAL) {
        float xd[L::VEC];
        L::unpack(rd, xd);
#pragma unroll
        for (int j = 0; j < L::VEC; ++j) {
            const float p = kept(xt[j], j, J.kt, J.it) ? ex2((xt[j] - J.mt) * J.c) * J.rzt : 0.0f;
            const float q = kept(xd[j], j, J.kd, J.id) ? ex2((xd[j] - J.md) * J.c) * J.rzd : 0.0f;
            w[j] = fmaxf(p - q, 0.0f);
        }
    } else {
#pragma unroll
        for (int j = 0; j < L::VEC; ++j)
            w[j] = kept(xt[j], j, J.kt, J.it) ? ex2((xt[j] - J.mt) * J.c) : 0.0f;
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

__device__ __forceinline__ JobRec load_job(const Params &P, int b)
{
    JobRec J;
    uint4 *dst = reinterpret_cast<uint4 *>(&J);
    const uint4 *src = reinterpret_cast<const uint4 *>(P.jobs + b);
#pragma unroll
    for (int i = 0; i < JOB_VECS; ++i)
        dst[i] = __ldg(src + i);
    return J;
}

// The inverse CDF's running mass C(x) is defined by a fixed hierarchy:
//   element -> lane (VEC elements, left to right) -> chunk (32 lanes,
//   Kogge-Stone) -> block (8 chunks, left to right) -> row (blocks, left to
//   right).  A block is NT vectors; chunk w of block k holds vectors
//   k*NT + 32*w .. k*NT + 32*w + 31.  A draw tile (one CTA) holds UD blocks;
//   warp w writes the totals of chunk w of each.
template <int DT, bool FILT>
__global__ void __launch_bounds__(NT, FILT ? 4 : 6) draw_kernel(const Params P)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    allow_next_kernel();
    wait_previous_kernel();  // the job comes from the scan kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // one draw tile per CTA, or (a grid smaller than the tiles) a stride over
    // them: when most sequences draw from their kept sets, launching a CTA
    // per tile costs more than the tiles left
    const unsigned int items = (unsigned int)P.DS * (unsigned int)P.B;
    if (FILT && P.gkey && __ldcg(&P.hdr->n_stream_draws) == 0u)
        return;  // every draw of the call comes from the kept sets
    for (unsigned int item = blockIdx.x; item < items; item += gridDim.x) {
        const int b = (int)(item / (unsigned int)P.DS);
        const int seg = (int)(item - (unsigned int)b * (unsigned int)P.DS);
        const JobRec J = load_job(P, b);
        if (J.mode == DRAW_NONE || (J.mode == DRAW_TARGET && !(FILT && J.filt)))
            continue;  // unfiltered bonus draws use the statistics kernel's chunk records
        if (FILT && J.pad0)
            continue;  // drawn from the kept sets (kdraw_kernel)
        float *out = P.chunks + (size_t)b * P.chunk_stride + (size_t)seg * UD * NCW;
        uint4 rt[UD], rd[UD];
#pragma unroll
        for (int u = 0; u < UD; ++u) {
            const int v = (seg * UD + u) * NT + warp * 32 + lane;
            rt[u] = row_vec<DT>(P.target, (size_t)J.t_row, v, P.V);
            rd[u] = (J.mode == DRAW_RESIDUAL) ? row_vec<DT>(P.draft, (size_t)J.d_row, v, P.V) : rt[u];
        }
        (void)VEC;
#pragma unroll
        for (int u = 0; u < UD; ++u) {
            float w[VEC];
            draw_weights<DT, FILT>(J, J.mode, rt[u], rd[u], w, ((seg * UD + u) * NT + warp * 32 + lane) * VEC);
            float tau = 0.0f;
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                tau = tau + w[j];
            float incl, excl;
            warp_scan(tau, lane, incl, excl);
            if (lane == 31)
                out[u * NCW + warp] = incl;
        }
    }
}

// ------------------------------------------- top-k draws from the kept sets
//
// A filtered sequence whose rows have top-k (K <= KF_KMAX) in a call with
// group maxima draws its correction or bonus token from the kept sets alone:
// the residual max(0, p~ - q~) and the bonus p~ are zero outside the target's
// kept set, which holds at most K tokens.  A kept set is read back as the
// group cut stored it (its tokens in rank order); for a row the cut left to
// the streaming filter it is gathered through the group maxima as the cut
// gathers them (the groups whose key is >= kappa; their tokens with key >
// kappa, or == kappa up to index iota), or, when more groups than the buffer
// holds reach kappa (ties), by a pass over the row.
// The weights are computed in fp64 as the fp64 reference computes them:
// exp((x - m) / T) over each kept set, normalised by its sum; the inverse CDF
// runs over the target's kept tokens in index order.
constexpr int KD_TH = 128;
constexpr int KD_CAP = 512;  // kept tokens at most (K <= KF_KMAX <= KD_CAP)
static_assert(KF_KMAX <= KD_CAP, "a kept set fits the buffer");

struct KdSmem {
    int gl[KF_GCAP];                   // groups reaching kappa
    int tidx[KD_CAP], didx[KD_CAP];    // kept tokens of the target / draft row
    float tval[KD_CAP], dval[KD_CAP];  // their logits
    double w[KD_CAP];                  // the target kept tokens' weights
    double ed[KD_CAP];                 // the draft kept tokens' exponentials
    int order[KD_CAP];                 // target kept tokens by index
    double red[KD_TH / 32];
    unsigned int ng, n;
};

// The kept set of one row into (oidx, oval); returns its size (every thread).
template <int DT>
__device__ int kd_gather(const Params &P, const void *arr, size_t row, const unsigned int *gk,
                         unsigned int kap, int iota, int *oidx, float *oval, KdSmem &S, int t,
                         int lane)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    constexpr int VPT = TILE_BYTES / 16;
    const size_t NG = (size_t)P.NS * NT;
    const int V = P.V;
    auto keep = [&](float x, int e) {
        const unsigned int key = key_of<DT>(x);
        return key > kap || (key == kap && e <= iota);
    };
    if (t == 0) {
        S.ng = 0u;
        S.n = 0u;
    }
    __syncthreads();
    // NG is a multiple of the block, so every lane takes each step; KF_LB key
    // loads in flight per thread
    for (size_t g0 = 0; g0 < NG; g0 += (size_t)KD_TH * KF_LB) {
        unsigned int key[KF_LB];
#pragma unroll
        for (int q = 0; q < KF_LB; ++q) {
            const size_t g = g0 + (size_t)q * KD_TH + t;
            key[q] = (g < NG) ? __ldcg(gk + g) : 0u;
        }
#pragma unroll
        for (int q = 0; q < KF_LB; ++q) {
            if (g0 + (size_t)q * KD_TH < NG) {  // the same in every lane
                const bool sel = key[q] >= kap;
                const unsigned int slot = warp_slot(sel, &S.ng, lane);
                if (sel && slot < (unsigned int)KF_GCAP)
                    S.gl[slot] = (int)(g0 + (size_t)q * KD_TH + t);
            }
        }
    }
    __syncthreads();
    const unsigned int ng = S.ng;
    if (ng <= (unsigned int)KF_GCAP) {
        const int nw = (int)ng * U;
        const bool aligned = ((row * (size_t)V) % VEC) == 0;
        for (int w0 = 0; w0 < nw; w0 += KD_TH) {  // every lane takes each step
            const int w = w0 + t;
            int v = -1;
            if (w < nw) {
                const int g = S.gl[w / U], u = w - (w / U) * U;
                const int seg = g / NT, gw = (g % NT) / 32, gl = g % 32;
                v = seg * VPT + 256 * gw + 32 * u + gl;
            }
            float x[VEC];
            if (v >= 0 && aligned && (v + 1) * VEC <= V) {
                L::unpack(__ldg(reinterpret_cast<const uint4 *>(arr) + (row * (size_t)V) / VEC + v),
                          x);
            } else {
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const int e = v * VEC + j;
                    x[j] = (v >= 0 && e < V) ? L::load1(arr, row * (size_t)V + e) : -INFINITY;
                }
            }
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const int e = v * VEC + j;
                const bool want = v >= 0 && e < V && keep(x[j], e);
                const unsigned int slot = warp_slot(want, &S.n, lane);
                if (want && slot < (unsigned int)KD_CAP) {
                    oidx[slot] = e;
                    oval[slot] = x[j];
                }
            }
        }
    } else {
        for (int e0 = 0; e0 < V; e0 += KD_TH) {  // every lane takes each step
            const int e = e0 + t;
            const float x = (e < V) ? L::load1(arr, row * (size_t)V + e) : -INFINITY;
            const bool want = e < V && keep(x, e);
            const unsigned int slot = warp_slot(want, &S.n, lane);
            if (want && slot < (unsigned int)KD_CAP) {
                oidx[slot] = e;
                oval[slot] = x;
            }
        }
    }
    __syncthreads();
    const int n = min((int)S.n, KD_CAP);
    __syncthreads();
    return n;
}

// The kept set of row `item` as the group cut stored it (rank order) into
// (oidx, oval); returns its size, or -1 when the cut left the row to the
// streaming filter (every thread).
template <int DT>
__device__ int kd_stored(const Params &P, size_t item, int *oidx, float *oval, int t)
{
    const int n = __ldcg(P.kcount + item);
    if (n < 0)
        return -1;
    const unsigned long long *kp = P.kept + item * KF_KMAX;
    for (int i = t; i < n; i += KD_TH) {
        const unsigned long long e = __ldcg(kp + i);
        oidx[i] = (int)(0xffffffffu - (unsigned int)(e & 0xffffffffu));
        oval[i] = val_of_key<DT>((unsigned int)(e >> 32));
    }
    __syncthreads();
    return n;
}

// Block-wide sum of one double per thread, in a fixed order (every thread).
__device__ __forceinline__ double kd_sum(double x, KdSmem &S, int t, int lane)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0)
        S.red[t >> 5] = x;
    __syncthreads();
    double s = 0.0;
    for (int w = 0; w < KD_TH / 32; ++w)
        s += S.red[w];
    __syncthreads();
    return s;
}

template <int DT>
__global__ void __launch_bounds__(KD_TH) kdraw_kernel(const Params P)
{
    using L = Lg<DT>;
    __shared__ KdSmem S;
    const int b = blockIdx.x;
    const int t = threadIdx.x, lane = t & 31;
    allow_next_kernel();
    wait_previous_kernel();  // the jobs come from the scan kernel (before the draw kernel)
    if (b >= P.B)
        return;
    const JobRec J = load_job(P, b);
    if (J.mode == DRAW_NONE || !J.filt || !J.pad0)
        return;
    const int k = P.k;
    const size_t NG = (size_t)P.NS * NT;
    const double T = (double)__ldg(P.temperature + b);
    const bool resid = J.mode == DRAW_RESIDUAL;
    // the target's kept set at row j (its bonus row when j == k): as the
    // group cut stored it, else gathered through the group maxima
    const size_t it_t = (size_t)b * P.rows + J.j;
    int nt = kd_stored<DT>(P, it_t, S.tidx, S.tval, t);
    if (nt < 0)
        nt = kd_gather<DT>(P, P.target, (size_t)J.t_row, P.gkey + it_t * NG, J.kt, J.it, S.tidx,
                           S.tval, S, t, lane);
    double zd = 1.0;
    int nd = 0;
    if (resid) {
        const size_t it_d = (size_t)b * P.rows + k + 1 + J.j;
        nd = kd_stored<DT>(P, it_d, S.didx, S.dval, t);
        if (nd < 0)
            nd = kd_gather<DT>(P, P.draft, (size_t)J.d_row, P.gkey + it_d * NG, J.kd, J.id,
                               S.didx, S.dval, S, t, lane);
        double z = 0.0;
        for (int i = t; i < nd; i += KD_TH) {
            const double e = exp(((double)S.dval[i] - (double)J.md) / T);
            S.ed[i] = e;
            z += e;
        }
        zd = kd_sum(z, S, t, lane);
    }
    // each exponential once (the fp64 pipe is narrow): the target's in S.w
    // until its weight replaces it, the draft's in S.ed
    double zt = 0.0;
    for (int i = t; i < nt; i += KD_TH) {
        const double e = exp(((double)S.tval[i] - (double)J.mt) / T);
        S.w[i] = e;
        zt += e;
    }
    zt = kd_sum(zt, S, t, lane);
    // weights of the target's kept tokens, and their order by index
    double r = 0.0;
    for (int i = t; i < nt; i += KD_TH) {
        const int x = S.tidx[i];
        const double p = S.w[i] / zt;
        double q = 0.0;
        if (resid) {
            // q~(x) is nonzero exactly when x is in the draft's kept set
            for (int j = 0; j < nd; ++j) {
                if (S.didx[j] == x) {
                    q = S.ed[j] / zd;
                    break;
                }
            }
        }
        const double w = resid ? fmax(p - q, 0.0) : p;
        S.w[i] = w;
        r += w;
        int rank = 0;
        for (int q2 = 0; q2 < nt; ++q2)
            rank += S.tidx[q2] < x ? 1 : 0;
        S.order[rank] = i;
    }
    const double R = kd_sum(r, S, t, lane);
    if (!(R > 0.0)) {
        // the residual vanished by rounding alone: draw from p~ instead
        for (int i = t; i < nt; i += KD_TH)
            S.w[i] = exp(((double)S.tval[i] - (double)J.mt) / T) / zt;
        __syncthreads();
    }
    if (t == 0) {
        double tot = 0.0;
        for (int q2 = 0; q2 < nt; ++q2)
            tot += S.w[S.order[q2]];
        const double target = (double)J.u * tot;
        double c = 0.0;
        int tok = -1, last = -1;
        for (int q2 = 0; q2 < nt; ++q2) {
            const int i = S.order[q2];
            if (S.w[i] > 0.0)
                last = S.tidx[i];
            c += S.w[i];
            if (c > target && S.w[i] > 0.0) {
                tok = S.tidx[i];
                break;
            }
        }
        if (tok < 0)
            tok = last;  // rounding left u * R at the total: the last positive weight
        P.out_tokens[(size_t)b * (k + 1) + J.j] = tok;
    }
}

// ------------------------------------------------------------- final search

// Totals of every block of one drawing sequence, then the crossing: block by
// block, then chunk by chunk, then within the chunk, C(x) = base + (W + (E +
// s)) with base the running block sum, W the running chunk sum in the block,
// E the lane's exclusive scan and s the lane's running sum.  The token is the
// smallest x with w(x) > 0 and C(x) > u * R, R the row total; if rounding
// leaves none in the chunk found, the chunk's last positive-weight token.
// Returns -1 when the total mass is zero.  `near` is set (every lane) when
// u * R lies within the guard of the chosen cell's edges, or a rounding
// fallback was taken: residual weights are probabilities, so their guard is
// absolute; target-row weights are unnormalised, so theirs is relative to R.
template <int DT, bool FILT>
__device__ int locate(const Params &P, const JobRec &J, int mode, const float *ch, float *btot,
                      int nblk, int lane, bool &near, float &gap_u)
{
    near = true;
    gap_u = 0.0f;
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    // block totals: 8 chunk totals left to right (two 16-byte loads per block,
    // four blocks per lane in flight)
    for (int blk0 = lane; blk0 < nblk; blk0 += 4 * 32) {
        float4 c8[4][NCW / 4];
#pragma unroll
        for (int g = 0; g < 4; ++g)
            if (blk0 + g * 32 < nblk)
#pragma unroll
                for (int w = 0; w < NCW / 4; ++w)
                    c8[g][w] = *reinterpret_cast<const float4 *>(ch + (blk0 + g * 32) * NCW + 4 * w);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (blk0 + g * 32 < nblk) {
                float bt = 0.0f;
#pragma unroll
                for (int w = 0; w < NCW / 4; ++w)
                    bt = (((bt + c8[g][w].x) + c8[g][w].y) + c8[g][w].z) + c8[g][w].w;
                btot[blk0 + g * 32] = bt;
            }
        }
    }
    __syncwarp();
    // the row level: an inclusive prefix of the block totals, left to right,
    // by one lane, carried as a float pair (each addition's rounding error is
    // kept and added back, so the running sum is good to about one rounding
    // whatever the number of blocks); then the first block whose prefix
    // exceeds u * R, found by the whole warp
    if (lane == 0) {
        float acc = 0.0f, err = 0.0f;
        auto add = [&](float x) {
            const float t = __fadd_rn(acc, x);
            const float bv = __fsub_rn(t, acc);
            err = __fadd_rn(err, __fadd_rn(__fsub_rn(acc, __fsub_rn(t, bv)), __fsub_rn(x, bv)));
            acc = t;
            return __fadd_rn(acc, err);
        };
        int blk = 0;
        for (; blk + 4 <= nblk; blk += 4) {
            const float4 t4 = *reinterpret_cast<const float4 *>(btot + blk);
            btot[blk] = add(t4.x);
            btot[blk + 1] = add(t4.y);
            btot[blk + 2] = add(t4.z);
            btot[blk + 3] = add(t4.w);
        }
        for (; blk < nblk; ++blk)
            btot[blk] = add(btot[blk]);
    }
    __syncwarp();
    const float R = btot[nblk - 1];
    if (!(R > 0.0f))
        return -1;
    const float uR = J.u * R;
    int bstar = nblk - 1;
    for (int blk0 = 0; blk0 < nblk; blk0 += 32) {
        const int blk = blk0 + lane;
        const unsigned hit = __ballot_sync(0xffffffffu, blk < nblk && btot[blk] > uR);
        if (hit) {
            bstar = blk0 + __ffs(hit) - 1;
            break;
        }
    }
    const float base = (bstar > 0) ? btot[bstar - 1] : 0.0f;
    const float cw = (lane < NCW) ? ch[bstar * NCW + lane] : 0.0f;
    float W = 0.0f;
    int wstar = NCW - 1;
    for (int w = 0; w < NCW; ++w) {
        const float nxt = W + __shfl_sync(0xffffffffu, cw, w);
        if (base + nxt > uR) {
            wstar = w;
            break;
        }
        W = nxt;
    }
    const int v = bstar * NT + wstar * 32 + lane;
    const uint4 rt = row_vec<DT>(P.target, (size_t)J.t_row, v, P.V);
    const uint4 rd = (mode == DRAW_RESIDUAL) ? row_vec<DT>(P.draft, (size_t)J.d_row, v, P.V) : rt;
    float w[VEC];
    draw_weights<DT, FILT>(J, mode, rt, rd, w, v * VEC);
    float sacc[VEC];
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        s = s + w[j];
        sacc[j] = s;
    }
    float incl, excl;
    warp_scan(s, lane, incl, excl);
    const float pre = W + excl;
    int cand = INT_MAX, lastp = -1;
    float gap = 0.0f;  // distance of u * R to the nearer edge of the lane's crossing cell
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        const int e = v * VEC + j;
        if (w[j] > 0.0f) {
            lastp = e;
            const float cur = base + (pre + sacc[j]);
            if (cand == INT_MAX && cur > uR) {
                cand = e;
                const float prev = base + (pre + (j > 0 ? sacc[j - 1] : 0.0f));
                gap = fminf(uR - prev, cur - uR);
            }
        }
    }
    const int mine = cand;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
        lastp = max(lastp, __shfl_xor_sync(0xffffffffu, lastp, o));
    }
    if (cand != INT_MAX) {
        const unsigned owner = __ballot_sync(0xffffffffu, mine == cand);
        gap = __shfl_sync(0xffffffffu, gap, __ffs(owner) - 1);
        const float guard = (mode == DRAW_RESIDUAL) ? P.guard_abs : P.guard_rel * R;
        near = !(gap >= guard);
        gap_u = gap / R;
    }
    return (cand != INT_MAX) ? cand : lastp;
}

// Chunk totals of a whole row computed by one warp (the rounding-only
// fallback when a residual vanished), in the same hierarchy as draw_kernel.
template <int DT, bool FILT>
__device__ void warp_row_chunks(const Params &P, const JobRec &J, int mode, float *ch, int nblk,
                                int lane)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    for (int blk = 0; blk < nblk; ++blk) {
        for (int w = 0; w < NCW; ++w) {
            const int v = blk * NT + w * 32 + lane;
            const uint4 rt = row_vec<DT>(P.target, (size_t)J.t_row, v, P.V);
            float x[VEC];
            draw_weights<DT, FILT>(J, mode, rt, rt, x, v * VEC);
            float tau = 0.0f;
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                tau = tau + x[j];
            float incl, excl;
            warp_scan(tau, lane, incl, excl);
            if (lane == 31)
                ch[blk * NCW + w] = incl;
        }
    }
    __syncwarp();
}

// The exact-draw record of a listed sequence (resolve.cuh).
template <int DT, bool FILT>
__device__ __forceinline__ RJob make_rjob(const Params &P, const JobRec &Jr, int b)
{
    RJob J;
    J.t_arr = P.target;
    J.d_arr = P.draft;
    J.t_row = Jr.t_row;
    J.d_row = Jr.d_row;
    J.mode = (Jr.mode == DRAW_RESIDUAL) ? RJ_RESIDUAL : RJ_TARGET;
    J.mt = Jr.mt;
    J.md = Jr.md;
    J.rzt = Jr.rzt;
    J.rzd = Jr.rzd;
    exp_coef(__ldg(P.temperature + b), J.ch, J.cl);
    J.u = Jr.u;
    J.filt = (FILT && Jr.filt) ? 1 : 0;
    J.kt = Jr.kt;
    J.it = Jr.it;
    J.kd = Jr.kd;
    J.id = Jr.id;
    J.b = b;
    J.out_pos = (long long)b * (P.k + 1) + Jr.j;
    return J;
}



template <int DT, bool FILT>
__global__ void __launch_bounds__(SCAN_WARPS * 32) final_kernel(const Params P)
{
    __shared__ float btot[SCAN_WARPS][MAXBLK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * SCAN_WARPS + warp;
    allow_next_kernel();     // the exact-draw kernel may launch; it waits for this grid
    wait_previous_kernel();  // chunk totals come from the draw kernel
    if (b >= P.B)
        return;
    const JobRec J = load_job(P, b);
    if (J.mode == DRAW_NONE)
        return;
    const int k = P.k;
    if (FILT && J.pad0) {
        // drawn from the kept sets: kdraw_kernel wrote out_tokens[b][j]
        for (int i = lane; i <= k; i += 32)
            if (i != J.j)
                P.out_tokens[(size_t)b * (k + 1) + i] =
                    (i < J.j) ? __ldg(P.tokens + (size_t)b * k + i) : -1;
        if (lane == 0)
            P.out_num_accepted[b] = J.j;
        return;
    }
    const int nblk = P.DS * UD;
    float *ch = P.chunks + (size_t)b * P.chunk_stride;
    int tok;
    bool near;
    float gap_u;  // the fp32 distance of u to the chosen cell's nearer edge (trace only)
    if (J.mode == DRAW_TARGET && !(FILT && J.filt))
        tok = records_draw<DT>(P.rec + (size_t)b * P.NCH, P.NCH, J.mt, J.c, J.u, P.target,
                               (size_t)J.t_row, P.V, lane, P.guard_rel, near, &gap_u);
    else
        tok = locate<DT, FILT>(P, J, J.mode, ch, btot[warp], nblk, lane, near, gap_u);
    if (tok < 0 && J.mode == DRAW_RESIDUAL) {
        // the residual vanished by rounding alone: draw from p_j instead
        warp_row_chunks<DT, FILT>(P, J, DRAW_TARGET, ch, nblk, lane);
        tok = locate<DT, FILT>(P, J, DRAW_TARGET, ch, btot[warp], nblk, lane, near, gap_u);
        near = true;
    }
    const bool err = tok < 0;
    if (!err && near && lane == 0) {
        // list the sequence for the exact draw, which rewrites out_tokens[b][j]
        const unsigned int f = atomicAdd(&P.hdr->n_flag, 1u);
        P.rjob[f] = make_rjob<DT, FILT>(P, J, b);
        P.rkcnt[f] = 0u;
    }
    if (P.out_draw && lane == 0) {
        P.out_draw[(size_t)b * 4 + 0] = tok;
        P.out_draw[(size_t)b * 4 + 1] = (!err && near) ? 1 : 0;
        P.out_draw[(size_t)b * 4 + 2] = tok;
        P.out_draw[(size_t)b * 4 + 3] = __float_as_int(gap_u);
    }
    for (int i = lane; i <= k; i += 32) {
        int o = -1;
        if (!err)
            o = (i < J.j) ? __ldg(P.tokens + (size_t)b * k + i) : (i == J.j ? tok : -1);
        P.out_tokens[(size_t)b * (k + 1) + i] = o;
    }
    if (lane == 0)
        P.out_num_accepted[b] = err ? -1 : J.j;
}

// ------------------------------------------------------------ exact draws
//
// The sequences final_kernel listed (their fp32 draw landed within the guard
// of a cell edge) are drawn again exactly (resolve.cuh).  Work items are
// (listed sequence, chunk of 2048 elements), dealt round robin over a
// persistent grid; the CTA that finishes a sequence's last chunk (a ticket
// counter, no waiting) forms the draw and rewrites out_tokens[b][j].

// ------------------------------------------------------------------ host side

// Per-device launch facts, filled by the first call on each device.  Host
// threads may call at once: a flag is published with release order after the
// values it guards, and read with acquire order (a race only repeats the same
// idempotent queries).
struct DevCache {
    std::atomic<int> sms;
    std::atomic<int> ctas_per_sm[2];     // statistics kernel, per dtype
    std::atomic<bool> attr_set[2];
    std::atomic<bool> filt_set[2];       // filter kernels' shared-memory sizes set
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
    size_t partials, jobs, chunks, rec, filt, resolve, total;
    size_t gkey, kept, kcount, total_filtered;  // filtered calls: the group-maximum regions
    size_t NS, NSS, DS, chunk_stride, NCH;
};

// header | one 16-byte partial per super-tile [B][2k+1][NSS] | draw jobs [B] |
// inverse-CDF chunk totals [B][chunk_stride] | bonus-row chunk records [B][NCH]
// | top-k / top-p records [B][2k+1] (filtered calls) | the exact draws of up
// to B listed sequences (resolve.cuh: records, counts, groups, chunk records)
// | and, when a filtered call's workspace has room, one 4-byte group key per
// 8 vectors of every tile of every row [B][2k+1][NS * 256], the kept tokens
// of the rows cut from them [B][2k+1][256] (8 bytes each) and their counts
// [B][2k+1]
WsLayout ws_layout(int32_t B, int32_t k, int32_t V, int32_t dtype)
{
    WsLayout w;
    const size_t te = tile_elems(dtype);
    const size_t es = (dtype == SPEC_F32) ? 4 : 2;
    w.NS = ((size_t)V + te - 1) / te;
    w.NSS = (w.NS + SUPER - 1) / SUPER;
    w.DS = ((size_t)V + te / 2 - 1) / (te / 2);
    w.NCH = ((size_t)V * es + CHUNK_BYTES - 1) / CHUNK_BYTES;
    w.partials = sizeof(WsHeader);
    w.jobs = align_up(w.partials + (size_t)B * (2 * (size_t)k + 1) * w.NSS * 16, 256);
    w.chunks = align_up(w.jobs + (size_t)B * sizeof(JobRec), 256);
    w.chunk_stride = align_up(w.DS * UD * NCW, 32);  // floats, 128-byte rows
    w.rec = align_up(w.chunks + (size_t)B * w.chunk_stride * 4, 256);
    w.filt = align_up(w.rec + (size_t)B * w.NCH * sizeof(float2), 256);
    w.resolve = align_up(w.filt + (size_t)B * (2 * (size_t)k + 1) * sizeof(FiltRec), 256);
    w.total = w.resolve + resolve_bytes((size_t)B, V, true);
    const size_t rows = (size_t)B * (2 * (size_t)k + 1);
    w.gkey = align_up(w.total, 256);
    w.kept = align_up(w.gkey + rows * w.NS * NT * 4, 256);
    w.kcount = align_up(w.kept + rows * KF_KMAX * 8, 256);
    w.total_filtered = w.kcount + rows * 4;
    return w;
}

size_t ws_bytes(int32_t B, int32_t k, int32_t V, int32_t dtype)
{
    return ws_layout(B, k, V, dtype).total;
}

// `events` (nullable): cudaEvent_t recorded after each kernel (five, or six
// with the filter kernels of a filtered call).
template <int DT, bool FILT>
int launch_all(const Params &P, const RParams &RP, unsigned int grid1, unsigned int gridf,
               unsigned int gridk, unsigned int gridk_draw, unsigned int gridr,
               unsigned int gridrf, cudaStream_t st, void *const *events)
{
    // filtered calls record one more event, after the filter kernel
    auto mark = [&](int i) {
        const int e = (FILT && i > 0) ? i + 1 : i;
        if (events && events[e])
            cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[e]), st);
    };
    // kernels 2..4 may start while their predecessor drains (programmatic
    // dependent launch); each waits before reading its predecessor's output.
    // With stage events requested, launches stay plainly ordered so each event
    // marks the end of its own stage.
    const bool pdl = !events;
    auto dependent = [&](auto kern, unsigned int grid, unsigned int block,
                         size_t smem = 0) -> cudaError_t {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(block);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, P);
    };
    stats_kernel<DT><<<grid1, NTHREADS, SMEM_BYTES, st>>>(P);
    mark(0);
    if constexpr (FILT) {
        // top-k rows are cut from the group maxima; the window kernel cuts
        // most other rows in one pass; the radix kernel finishes the rows
        // either of them flagged
        if (P.gkey && dependent(kfilter_kernel<DT>, gridk, KF_TH) != cudaSuccess)
            return SPEC_ECUDA;
        if (dependent(wfilter_kernel<DT>, gridf, WTH, WFILT_SMEM) != cudaSuccess)
            return SPEC_ECUDA;
        if (dependent(filter_kernel<DT>, gridf, FTH, FILT_SMEM) != cudaSuccess)
            return SPEC_ECUDA;
        if (events && events[1])
            cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[1]), st);
    }
    const unsigned int gs = (unsigned int)((P.B + SCAN_WARPS - 1) / SCAN_WARPS);
    if (dependent(scan_kernel<DT, FILT>, gs, SCAN_WARPS * 32) != cudaSuccess)
        return SPEC_ECUDA;
    mark(1);
    const unsigned int draw_tiles = (unsigned int)P.DS * (unsigned int)P.B;
    const unsigned int gridd = (FILT && P.gkey && draw_tiles > gridk_draw) ? gridk_draw : draw_tiles;
    if (dependent(draw_kernel<DT, FILT>, gridd, NT) != cudaSuccess)
        return SPEC_ECUDA;
    if constexpr (FILT) {
        if (P.gkey && dependent(kdraw_kernel<DT>, (unsigned int)P.B, KD_TH) != cudaSuccess)
            return SPEC_ECUDA;
    }
    mark(2);
    if (dependent(final_kernel<DT, FILT>, gs, SCAN_WARPS * 32) != cudaSuccess)
        return SPEC_ECUDA;
    mark(3);
    if (launch_resolve<DT>(RP, gridr, gridrf, st, pdl) != cudaSuccess)
        return SPEC_ECUDA;
    mark(4);
    if (cudaPeekAtLastError() != cudaSuccess) {
        (void)cudaGetLastError();
        return SPEC_ECUDA;
    }
    return SPEC_OK;
}

// Guards of the fp32 draw, below which a draw is redone exactly.  The fp32
// edges of a cell (ex2.approx weights, fp32 masses and chunk sums, the
// compensated running sum over blocks) were measured against the fp64
// oracle over ~5900 draws of the synthetic workloads: residual draws within
// 1.7e-7 in probability units (their weights are probabilities, so their
// guard is absolute), target-row draws within 3e-7 of R (relative).  The
// guards leave a factor of 4.
constexpr float GUARD_ABS = 7e-7f;
constexpr float GUARD_REL = 1.2e-6f;

int launch(const void *target, const void *draft, const int32_t *tokens, const float *ua,
           const float *ur, const float *temp, int32_t *out_tokens, int32_t *out_n,
           float *out_probs, int32_t B, int32_t k, int32_t V, int32_t dtype, void *ws,
           size_t ws_size, void *stream, void *const *events = nullptr, bool filtered = false,
           const int32_t *top_k = nullptr, const float *top_p = nullptr,
           int32_t *out_draw = nullptr, bool resolve_all = false)
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
        (reinterpret_cast<uintptr_t>(out_n) & 3) || (reinterpret_cast<uintptr_t>(out_probs) & 3) ||
        (reinterpret_cast<uintptr_t>(top_k) & 3) || (reinterpret_cast<uintptr_t>(top_p) & 3))
        return SPEC_EINVAL;
    const WsLayout lay = ws_layout(B, k, V, dtype);
    if (ws_size < lay.total)
        return SPEC_ENOSPACE;
    const size_t total = (size_t)B * (2 * (size_t)k + 1) * lay.NSS;
    if (total >= 0x7fffffffull || (size_t)B * lay.DS >= 0x7fffffffull)
        return SPEC_EINVAL;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SPEC_ECUDA;
    DevCache &dc = g_dev[dev];
    const int di = (dtype == SPEC_F32) ? 0 : 1;
    const void *fn = (dtype == SPEC_F32) ? (const void *)stats_kernel<SPEC_F32>
                                         : (const void *)stats_kernel<SPEC_BF16>;
    if (!dc.attr_set[di].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_BYTES) != cudaSuccess)
            return SPEC_ECUDA;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, NTHREADS, SMEM_BYTES) != cudaSuccess)
            return SPEC_ECUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SPEC_ECUDA;
        dc.sms.store(sms, std::memory_order_relaxed);
        dc.ctas_per_sm[di].store(n > 0 ? n : 1, std::memory_order_relaxed);
        dc.attr_set[di].store(true, std::memory_order_release);
    }
    const size_t n_sms = (size_t)dc.sms.load(std::memory_order_relaxed);
    unsigned int gridf = 0;
    if (filtered) {
        if (!dc.filt_set[di].load(std::memory_order_acquire)) {
            const void *ff = (dtype == SPEC_F32) ? (const void *)filter_kernel<SPEC_F32>
                                                 : (const void *)filter_kernel<SPEC_BF16>;
            if (cudaFuncSetAttribute(ff, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)FILT_SMEM) != cudaSuccess)
                return SPEC_ECUDA;
            const void *fw = (dtype == SPEC_F32) ? (const void *)wfilter_kernel<SPEC_F32>
                                                 : (const void *)wfilter_kernel<SPEC_BF16>;
            if (cudaFuncSetAttribute(fw, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)WFILT_SMEM) != cudaSuccess)
                return SPEC_ECUDA;
            dc.filt_set[di].store(true, std::memory_order_release);
        }
        // two rows per SM in flight (one CTA each, streaming through a ring)
        const size_t rows = (size_t)B * (2 * (size_t)k + 1);
        const size_t cap = n_sms * 2;
        gridf = (unsigned int)(rows < cap ? rows : cap);
    }
    const size_t resident = n_sms * (size_t)dc.ctas_per_sm[di].load(std::memory_order_relaxed);
    const unsigned int grid1 = (unsigned int)(total < resident ? total : resident);

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
    uint8_t *w = reinterpret_cast<uint8_t *>(ws);
    P.hdr = reinterpret_cast<WsHeader *>(w);
    P.part = reinterpret_cast<float4 *>(w + lay.partials);
    P.jobs = reinterpret_cast<JobRec *>(w + lay.jobs);
    P.chunks = reinterpret_cast<float *>(w + lay.chunks);
    P.rec = reinterpret_cast<float2 *>(w + lay.rec);
    P.top_k = top_k;
    P.top_p = top_p;
    P.filt = reinterpret_cast<FiltRec *>(w + lay.filt);
    const bool groups = filtered && ws_size >= lay.total_filtered;
    P.gkey = groups ? reinterpret_cast<unsigned int *>(w + lay.gkey) : nullptr;
    P.kept = groups ? reinterpret_cast<unsigned long long *>(w + lay.kept) : nullptr;
    P.kcount = groups ? reinterpret_cast<int *>(w + lay.kcount) : nullptr;
    RParams RP;
    resolve_regions(RP, w + lay.resolve, (size_t)B, V, true);
    RP.hdr = P.hdr;
    RP.out = out_tokens;
    RP.out_draw = out_draw;
    P.rjob = const_cast<RJob *>(RP.rjob);
    P.rkcnt = RP.rkcnt;
    P.guard_abs = resolve_all ? INFINITY : GUARD_ABS;
    P.guard_rel = resolve_all ? INFINITY : GUARD_REL;
    P.out_draw = out_draw;
    P.NCH = (int)lay.NCH;
    P.B = B;
    P.k = k;
    P.V = V;
    P.NS = (int)lay.NS;
    P.NSS = (int)lay.NSS;
    P.rows = 2 * k + 1;
    P.DS = (int)lay.DS;
    P.chunk_stride = (int)lay.chunk_stride;
    P.total_super = (unsigned int)total;
    const size_t es = (dtype == SPEC_F32) ? 4 : 2;
    P.target_bytes = (unsigned long long)B * (k + 1) * (unsigned long long)V * es;
    P.draft_bytes = (unsigned long long)B * k * (unsigned long long)V * es;

    // the exact draws: two CTAs per SM, at most one work item each to begin with
    const size_t ritems = (size_t)B * (size_t)RP.RNC;
    const unsigned int gridr = (unsigned int)(ritems < 3 * n_sms ? ritems : 3 * n_sms);
    const unsigned int gridrf = (unsigned int)((size_t)B < n_sms ? (size_t)B : n_sms);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the group-maximum cut: sixteen CTAs of 128 threads per SM (a full SM;
    // its 12 KB of shared memory allow it), rows dealt round robin
    const size_t nrows = (size_t)B * (2 * (size_t)k + 1);
    const unsigned int gridk = (unsigned int)(nrows < 16 * n_sms ? nrows : 16 * n_sms);
    // with kept-set draws, the draw kernel strides over its tiles with the
    // CTAs that fit at once (four per SM)
    const unsigned int gridk_draw = (unsigned int)(4 * n_sms);
    if (filtered)
        return (dtype == SPEC_F32)
                   ? launch_all<SPEC_F32, true>(P, RP, grid1, gridf, gridk, gridk_draw, gridr, gridrf,
                                                st, events)
                   : launch_all<SPEC_BF16, true>(P, RP, grid1, gridf, gridk, gridk_draw, gridr, gridrf,
                                                 st, events);
    return (dtype == SPEC_F32)
               ? launch_all<SPEC_F32, false>(P, RP, grid1, 0, 0, 0, gridr, gridrf, st, events)
               : launch_all<SPEC_BF16, false>(P, RP, grid1, 0, 0, 0, gridr, gridrf, st, events);
}

}  // namespace

static_assert(SPEC_MAX_V / (NT * 4) + UD <= MAXBLK, "CDF blocks must cover the largest vocabulary");

// ------------------------------------------------- scratch without allocation
//
// Device-resident scratch for spec_verify_noalloc.  It is part of the loaded
// module: every GPU that loads this library holds these bytes until the
// process exits.  Host code must not pass the symbol itself to a kernel (on
// the host it names a host-side stand-in); the device address comes from
// cudaGetSymbolAddress, once per device, with that device current.
constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)8 << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];
static std::atomic<void *> g_noalloc_addr[64];

namespace spec_internal {

// The scratch array's device address on the current device: looked up the
// first time (cudaGetSymbolAddress, with that device current) and kept.
int noalloc_scratch(void **addr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SPEC_ECUDA;
    void *ws = g_noalloc_addr[dev].load(std::memory_order_relaxed);
    if (!ws) {
        if (cudaGetSymbolAddress(&ws, g_noalloc_scratch) != cudaSuccess || !ws)
            return SPEC_ECUDA;
        g_noalloc_addr[dev].store(ws, std::memory_order_relaxed);
    }
    *addr = ws;
    return SPEC_OK;
}

}  // namespace spec_internal

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

size_t spec_verify_filtered_workspace_size(int32_t B, int32_t k, int32_t V, int32_t dtype)
{
    if (!sizes_ok(B, k, V, dtype))
        return 0;
    return ws_layout(B, k, V, dtype).total_filtered;
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

int32_t spec_verify_filtered(const void *target_logits, const void *draft_logits,
                             const int32_t *draft_tokens, const float *u_accept,
                             const float *u_resample, const float *temperature,
                             const int32_t *top_k, const float *top_p,
                             int32_t *out_tokens, int32_t *out_num_accepted, float *out_probs,
                             int32_t B, int32_t k, int32_t V, int32_t dtype,
                             void *workspace, size_t workspace_bytes, void *stream)
{
    return launch(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature,
                  out_tokens, out_num_accepted, out_probs, B, k, V, dtype, workspace,
                  workspace_bytes, stream, nullptr, true, top_k, top_p);
}

int32_t spec_verify_filtered_timed(const void *target_logits, const void *draft_logits,
                                   const int32_t *draft_tokens, const float *u_accept,
                                   const float *u_resample, const float *temperature,
                                   const int32_t *top_k, const float *top_p,
                                   int32_t *out_tokens, int32_t *out_num_accepted,
                                   int32_t B, int32_t k, int32_t V, int32_t dtype,
                                   void *workspace, size_t workspace_bytes, void *stream,
                                   void *const *stage_events)
{
    return launch(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature,
                  out_tokens, out_num_accepted, nullptr, B, k, V, dtype, workspace,
                  workspace_bytes, stream, stage_events, true, top_k, top_p);
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

int32_t spec_verify_trace(const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *u_accept,
                          const float *u_resample, const float *temperature,
                          int32_t *out_tokens, int32_t *out_num_accepted, float *out_probs,
                          int32_t *out_draw, int32_t resolve_all,
                          int32_t B, int32_t k, int32_t V, int32_t dtype,
                          void *workspace, size_t workspace_bytes, void *stream)
{
    if (!out_draw && B > 0)
        return SPEC_EINVAL;
    if (reinterpret_cast<uintptr_t>(out_draw) & 3)
        return SPEC_EINVAL;
    return launch(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature,
                  out_tokens, out_num_accepted, out_probs, B, k, V, dtype, workspace,
                  workspace_bytes, stream, nullptr, false, nullptr, nullptr, out_draw,
                  resolve_all != 0);
}

int32_t spec_verify_timed(const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *u_accept,
                          const float *u_resample, const float *temperature,
                          int32_t *out_tokens, int32_t *out_num_accepted,
                          int32_t B, int32_t k, int32_t V, int32_t dtype,
                          void *workspace, size_t workspace_bytes, void *stream,
                          void *const *stage_events)
{
    return launch(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature,
                  out_tokens, out_num_accepted, nullptr, B, k, V, dtype, workspace,
                  workspace_bytes, stream, stage_events);
}

int32_t spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                            const int32_t *draft_tokens, const float *u_accept,
                            const float *u_resample, const float *temperature,
                            int32_t *out_tokens, int32_t *out_num_accepted,
                            int32_t B, int32_t k, int32_t V, int32_t dtype, void *stream)
{
    if (!sizes_ok(B, k, V, dtype))
        return SPEC_EINVAL;
    if (B == 0)
        return SPEC_OK;
    if (ws_bytes(B, k, V, dtype) > NOALLOC_SCRATCH_BYTES)
        return SPEC_ENOSPACE;
    void *ws = nullptr;
    const int rc = spec_internal::noalloc_scratch(&ws);
    if (rc != SPEC_OK)
        return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the status word is the only scratch contents a call reads before writing
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), st) != cudaSuccess)
        return SPEC_ECUDA;
    return launch(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature,
                  out_tokens, out_num_accepted, nullptr, B, k, V, dtype, ws,
                  NOALLOC_SCRATCH_BYTES, stream);
}

size_t spec_verify_noalloc_max_bytes(void) { return NOALLOC_SCRATCH_BYTES; }

int32_t spec_verify_noalloc_read_status(int32_t *status, void *stream)
{
    if (!status)
        return SPEC_EINVAL;
    void *ws = nullptr;
    const int rc = spec_internal::noalloc_scratch(&ws);
    if (rc != SPEC_OK)
        return rc;
    return spec_verify_read_status(ws, status, stream);
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
    } cps[] = {{d_t, target_logits, bt},
               {d_g, draft_tokens, (size_t)B * k * 4}, {d_ua, u_accept, (size_t)B * k * 4},
               {d_ur, u_resample, (size_t)B * 4},    {d_T, temperature, (size_t)B * 4}};
    for (const auto &c : cps)
        if (cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return SPEC_ECUDA;
    // A greedy sequence's draft rows are never read (the greedy rule compares
    // argmaxes of the target alone), so only the other sequences' draft rows
    // cross the host link: one copy per run of consecutive such sequences.
    const size_t drow = (size_t)k * V * es;
    for (int b0 = 0; b0 < B;) {
        if (temperature[b0] == 0.0f) {
            ++b0;
            continue;
        }
        int b1 = b0 + 1;
        while (b1 < B && !(temperature[b1] == 0.0f))
            ++b1;
        if (cudaMemcpyAsync(d_d + (size_t)b0 * drow,
                            reinterpret_cast<const uint8_t *>(draft_logits) + (size_t)b0 * drow,
                            (size_t)(b1 - b0) * drow, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return SPEC_ECUDA;
        b0 = b1;
    }
    if (cudaMemsetAsync(d_ws, 0, sizeof(WsHeader), st) != cudaSuccess)
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
