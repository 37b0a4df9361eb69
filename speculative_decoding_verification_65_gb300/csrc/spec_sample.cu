// spec_sample.cu -- GB300 (sm_103a) kernels and C ABI for batched token
// sampling: one token per row from softmax(logits / T) by inverse CDF with a
// caller uniform (the draft model's sampling step, "Speculative Decoding and
// the Art of Fast LLM Inference", "The Algorithm, Step by Step"; the
// techaiinterview answer, "Algorithm (one round)", step 1).
//
// Every logit is read from HBM once.  Two kernels run on the caller's stream:
//   1. chunk_kernel: persistent and warp-specialised like the verification's
//      statistics kernel.  A producer warp deals groups of four consecutive
//      32 KB tiles of a row round robin over CTAs and streams the tiles with
//      cp.async.bulk into a 3-stage
//      shared-memory ring (mbarriers, bounded waits).  Consumer warp w owns the
//      contiguous 4 KB chunk w of each tile (lane l reads the 16-byte vectors
//      256*w + 32*u + l, u < 8) and writes one 8-byte record per chunk:
//      (chunk maximum M, sum of 2^((x - M) * c)) for a sampled row, with
//      c = log2(e) / T, or (M, lowest index attaining it) for a greedy row.
//      A lane sums 2^((x - m_l) * c) against its own maximum m_l and scales
//      the sum by 2^((m_l - M) * c) once, after the warp maximum is known.
//   2. pick_kernel: one warp per row.  It folds the records into the row
//      maximum m, scales each chunk's sum by 2^((M - m) * c), takes running
//      totals (each lane a contiguous range of chunks, then a Kogge-Stone scan
//      over lanes) up to R, finds the chunk whose total crosses u * R, reads
//      that one chunk again and searches it in index order (vectors u = 0..7
//      of the chunk, a Kogge-Stone scan over the 32 lanes of each, elements
//      left to right in a lane).
// The first kernel sums each lane's exponentials relative to the lane's own
// maximum and rescales the lane sums to the chunk maximum; the search takes
// them relative to the chunk maximum directly.  The two agree to fp32
// rounding, and a threshold that rounding leaves past the chunk's last running
// total takes the chunk's last positive weight -- the clamp the method's
// reading already has for the whole row.
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "spec_sample.h"
#include "internal.h"
#include "spec_verify.h"
#include "device_common.cuh"
#include "resolve.cuh"

namespace {

using namespace spec_dev;

constexpr int NCW = 8;                           // consumer warps
constexpr int WARP_P = NCW;                      // producer warp
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int STAGES = 3;
constexpr int TILE_BYTES = 32768;
constexpr int SLOT_BYTES = TILE_BYTES + 128;     // room for a misaligned head/tail
constexpr int UV = CHUNK_UV;                     // vectors per lane per chunk
constexpr int PICK_WARPS = 8;                    // rows per CTA of the pick kernel
constexpr int GROUP = 8;                         // consecutive tiles of a row per deal

static_assert(NCW * CHUNK_BYTES == TILE_BYTES, "a tile is one chunk per consumer warp");

enum { KIND_END = 0, KIND_TILE = 1 };
enum { MODE_GREEDY = 1, MODE_SAMPLE = 2 };

struct TileInfo {
    int kind;
    int row;
    int seg;      // tile of the row
    int mode;
    float c;      // log2(e) / T
    int phase0;   // bytes from the copy start to the tile's first element
    int ncopied0; // bytes present in the slot
    int pad;
};

struct SParams {
    const void *logits;
    const float *u;
    const float *temperature;
    int32_t *out;
    WsHeader *hdr;
    float2 *rec;       // [R][NC] chunk records
    int R, V;
    int NS;            // tiles per row
    int NC;            // chunks per row
    int NG;            // groups of GROUP tiles per row
    unsigned int total_groups;
    unsigned long long bytes;
    int rows_per_temp;  // row r's temperature is temperature[r / rows_per_temp]
    int skip_greedy;    // rows at T = 0 are not read (their records are not used)
    // the exact draw of rows whose fp32 draw lands near a cell edge
    RJob *rjob;          // [R] the listed rows (count in hdr->n_flag)
    unsigned int *rkcnt; // [R]
    float guard;         // list when u*R is within guard*R of a cell edge
};

struct Smem {
    unsigned long long full[STAGES];
    unsigned long long empty[STAGES];
    TileInfo info[STAGES];
    float tabT[32];    // the producer's temperatures for its next 32 groups
};

constexpr size_t SMEM_BYTES = (size_t)STAGES * SLOT_BYTES + sizeof(Smem);

// ----------------------------------------------------------- chunk records

template <int DT>
__global__ void __launch_bounds__(NTHREADS, 2) chunk_kernel(const SParams P)
{
    using L = Lg<DT>;
    constexpr int VEC = L::VEC;
    constexpr int SEG = TILE_BYTES / L::ES;  // elements per tile
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *slots = smem_raw;
    Smem &S = *reinterpret_cast<Smem *>(smem_raw + (size_t)STAGES * SLOT_BYTES);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        if (blockIdx.x == 0) {  // the exact draws' counters (used after this grid)
            P.hdr->n_flag = 0u;
            P.hdr->next_resolve = 0u;
        }
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], NCW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    allow_next_kernel();

    if (warp == WARP_P) {
        // ------------------------------------------------------- producer
        int stage = 0;
        uint32_t phase = 0;
        int issued_phase[STAGES];
        for (int s = 0; s < STAGES; ++s)
            issued_phase[s] = -1;
        int ok = 1;
        const unsigned int G = gridDim.x;
        // groups of GROUP consecutive tiles of one row are dealt round robin
        for (unsigned int base = blockIdx.x; base < P.total_groups && ok; base += 32u * G) {
            // each lane fetches the temperature of one of the next 32 groups
            const unsigned long long gl = base + (unsigned long long)lane * G;
            const float Tl = (gl < P.total_groups)
                                 ? __ldg(P.temperature + gl / (unsigned int)P.NG /
                                                             (unsigned int)P.rows_per_temp)
                                 : 0.0f;
            __syncwarp();  // lane 0 is done with the previous batch
            S.tabT[lane] = Tl;
            __syncwarp();
            if (lane == 0) {
                for (int i = 0; i < 32 && ok; ++i) {
                    const unsigned long long gi = base + (unsigned long long)i * G;
                    if (gi >= P.total_groups)
                        break;
                    const float T = S.tabT[i];
                    if (!temperature_valid(T) || (P.skip_greedy && T == 0.0f))
                        continue;  // nobody reads this row's records
                    const int row = (int)(gi / (unsigned int)P.NG);
                    const int grp = (int)(gi - (unsigned long long)row * (unsigned int)P.NG);
                    const int seg1 = min(P.NS, (grp + 1) * GROUP);
                    for (int seg = grp * GROUP; seg < seg1; ++seg) {
                        if (!mbar_wait(&S.empty[stage], phase ^ 1u)) {
                            atomicExch(&P.hdr->status, SPEC_DEV_WAIT_TIMEOUT);
                            ok = 0;
                            break;
                        }
                        TileInfo &ti = S.info[stage];
                        ti.kind = KIND_TILE;
                        ti.row = row;
                        ti.seg = seg;
                        ti.mode = (T == 0.0f) ? MODE_GREEDY : MODE_SAMPLE;
                        ti.c = (T == 0.0f) ? 0.0f : LOG2E / T;
                        const int e0 = seg * SEG, e1 = min(P.V, e0 + SEG);
                        const unsigned long long start =
                            ((unsigned long long)row * P.V + e0) * L::ES;
                        const unsigned long long end = ((unsigned long long)row * P.V + e1) * L::ES;
                        const unsigned long long a0 = start & ~15ull;
                        unsigned long long a1 = (end + 15) & ~15ull;
                        if (a1 > (P.bytes & ~15ull))
                            a1 = P.bytes & ~15ull;
                        const uint32_t bytes = (a1 > a0) ? (uint32_t)(a1 - a0) : 0u;
                        ti.phase0 = (int)(start - a0);
                        ti.ncopied0 = (int)bytes;
                        if (bytes) {
                            mbar_arrive_expect_tx(&S.full[stage], bytes);
                            bulk_copy_g2s(slots + (size_t)stage * SLOT_BYTES,
                                          reinterpret_cast<const uint8_t *>(P.logits) + a0, bytes,
                                          &S.full[stage]);
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
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        if (lane != 0)
            return;
        if (ok) {
            if (mbar_wait(&S.empty[stage], phase ^ 1u)) {
                S.info[stage].kind = KIND_END;
                mbar_arrive(&S.full[stage]);
            } else {
                atomicExch(&P.hdr->status, SPEC_DEV_WAIT_TIMEOUT);
                ok = 0;
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
        const int e0 = ti.seg * SEG, e1 = min(P.V, e0 + SEG);
        const int chunk = ti.seg * NCW + warp;  // chunk index within the row
        if (chunk < P.NC) {
            const Seg g = make_seg<DT>(slot, P.logits, (size_t)ti.row, P.V, e0, e1, ti.phase0,
                                       ti.ncopied0);
            const int vb = e0 / VEC + warp * (32 * UV);  // row-relative first vector of the chunk
            uint4 raw[UV];
            if (g.fast && e1 - e0 == SEG) {
#pragma unroll
                for (int u = 0; u < UV; ++u)
                    raw[u] = ld_shared_v4(slot + (size_t)(warp * 32 * UV + u * 32 + lane) * 16);
            } else {
#pragma unroll
                for (int u = 0; u < UV; ++u)
                    raw[u] = seg_vec<DT>(g, vb + u * 32 + lane);
            }
            float M, second;
            if (ti.mode == MODE_GREEDY) {
                float vmax[UV];
#pragma unroll
                for (int u = 0; u < UV; ++u)
                    vmax[u] = L::vmax(raw[u]);
                float ml = vmax[0];
#pragma unroll
                for (int u = 1; u < UV; ++u)
                    ml = fmax_nan(ml, vmax[u]);
                M = ml;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    M = fmax_nan(M, __shfl_xor_sync(0xffffffffu, M, o));
                // lowest index attaining M: this lane's earliest, then the warp's
                int idx = INT_MAX;
#pragma unroll
                for (int u = 0; u < UV; ++u) {
                    if (idx == INT_MAX && vmax[u] == M) {
                        float x[VEC];
                        L::unpack(raw[u], x);
#pragma unroll
                        for (int j = VEC - 1; j >= 0; --j)
                            if (x[j] == M)
                                idx = (vb + u * 32 + lane) * VEC + j;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
                second = __int_as_float(idx);
            } else {
                // exponentials relative to the lane's own maximum, so they need
                // no warp-wide value; the lane sums are rescaled to the chunk
                // maximum at the end
                const float ml = L::tile_max(raw);
                float s = 0.0f;
                if (ml != -INFINITY) {
                    const unsigned long long c2 = f2(ti.c, ti.c);
                    unsigned long long acc = L::expsum2(raw[0], -ml, c2);
#pragma unroll
                    for (int u = 1; u < UV; ++u)
                        acc = add2(acc, L::expsum2(raw[u], -ml, c2));
                    float s0, s1;
                    f2_split(acc, s0, s1);
                    s = s0 + s1;
                }
                M = ml;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    M = fmax_nan(M, __shfl_xor_sync(0xffffffffu, M, o));
                s = rescale(s, ml, M, ti.c);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    s += __shfl_xor_sync(0xffffffffu, s, o);
                second = s;
            }
            if (lane == 0)
                __stcg(P.rec + (size_t)ti.row * P.NC + chunk, make_float2(M, second));
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&S.empty[stage]);
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

// -------------------------------------------------------------------- pick

template <int DT>
__global__ void __launch_bounds__(PICK_WARPS * 32) pick_kernel(const SParams P)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * PICK_WARPS + warp;
    if (r >= P.R)
        return;
    const float T = __ldg(P.temperature + r);
    const float uu = __ldg(P.u + r);
    allow_next_kernel();
    wait_previous_kernel();  // the records come from the chunk kernel
    if (!temperature_valid(T)) {
        if (lane == 0)
            P.out[r] = -1;
        return;
    }
    const bool greedy = (T == 0.0f);
    const float c = greedy ? 0.0f : LOG2E / T;
    const float2 *rc = P.rec + (size_t)r * P.NC;
    const int per = (P.NC + 31) / 32;
    const int c0 = min(P.NC, lane * per), c1 = min(P.NC, c0 + per);

    // 1. row maximum (and, greedy, the earliest chunk holding it)
    float ml = -INFINITY;
    int il = INT_MAX;
    for (int q = c0; q < c1; ++q) {
        const float2 f = __ldcg(rc + q);
        if (f.x > ml && greedy)
            il = __float_as_int(f.y);
        ml = fmax_nan(ml, f.x);
    }
    float m = ml;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (isnan(m) || isinf(m)) {  // NaN, +inf, or every logit -inf
        if (lane == 0)
            P.out[r] = -1;
        return;
    }
    if (greedy) {
        int cand = (ml == m) ? il : INT_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
        if (lane == 0)
            P.out[r] = cand;
        return;
    }

    bool near = false;
    const int tok = records_draw<DT>(rc, P.NC, m, c, uu, P.logits, (size_t)r, P.V, lane, P.guard, near);
    if (lane == 0) {
        P.out[r] = tok;
        if (near && tok >= 0 && P.rjob) {
            // list the row for the exact draw (resolve.cuh), which rewrites out[r]
            const unsigned int f = atomicAdd(&P.hdr->n_flag, 1u);
            RJob J;
            J.t_arr = J.d_arr = P.logits;
            J.t_row = J.d_row = r;
            J.mode = RJ_TARGET;
            J.mt = J.md = m;
            J.rzt = J.rzd = 1.0f;
            exp_coef(T, J.ch, J.cl);
            J.u = uu;
            J.filt = 0;
            J.kt = J.kd = 0u;
            J.it = J.id = 0;
            J.b = r;
            J.out_pos = r;
            P.rjob[f] = J;
            P.rkcnt[f] = 0u;
        }
    }
}

// --------------------------------------------------------------- host side

// Per-device launch facts, filled by the first call on each device; the flag
// is published with release order after the values (host threads may race
// here, repeating the same idempotent queries).
struct DevCache {
    std::atomic<int> sms;
    std::atomic<int> ctas_per_sm[2];
    std::atomic<bool> attr_set[2];
};
DevCache g_dev[64];

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool sizes_ok(int32_t R, int32_t V, int32_t dtype)
{
    return R >= 0 && V >= 2 && V <= SPEC_MAX_V && (dtype == SPEC_F32 || dtype == SPEC_BF16);
}

struct Layout {
    size_t rec, resolve, total;
    size_t NS, NC;
};

// header | chunk records [R][NC] | the exact draws of up to R listed rows
// (resolve.cuh)
Layout layout(int32_t R, int32_t V, int32_t dtype)
{
    Layout w;
    const size_t es = (dtype == SPEC_F32) ? 4 : 2;
    const size_t row_bytes = (size_t)V * es;
    w.NS = (row_bytes + TILE_BYTES - 1) / TILE_BYTES;
    w.NC = (row_bytes + CHUNK_BYTES - 1) / CHUNK_BYTES;
    w.rec = sizeof(WsHeader);
    w.resolve = align_up(w.rec + (size_t)R * w.NC * sizeof(float2), 256);
    w.total = w.resolve + resolve_bytes((size_t)R, V, false);
    return w;
}

template <int DT>
int launch_all(const SParams &P, const RParams &RP, unsigned int gridr, unsigned int gridrf,
               unsigned int grid1, cudaStream_t st, void *const *events)
{
    auto mark = [&](int i) {
        if (events && events[i])
            cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), st);
    };
    chunk_kernel<DT><<<grid1, NTHREADS, SMEM_BYTES, st>>>(P);
    mark(0);
    // the pick kernel may start while the chunk kernel drains (programmatic
    // dependent launch); it waits before reading the records.  Plain order
    // when stage events are requested.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned int)((P.R + PICK_WARPS - 1) / PICK_WARPS));
    cfg.blockDim = dim3(PICK_WARPS * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = events ? 0 : 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, pick_kernel<DT>, P) != cudaSuccess)
        return SPEC_ECUDA;
    mark(1);
    if (launch_resolve<DT>(RP, gridr, gridrf, st, !events) != cudaSuccess)
        return SPEC_ECUDA;
    mark(2);
    if (cudaPeekAtLastError() != cudaSuccess) {
        (void)cudaGetLastError();
        return SPEC_ECUDA;
    }
    return SPEC_OK;
}

// The chunk kernel's parameters and grid for R rows of V logits; the
// records go to `rec`, the status to `hdr`.
int setup_chunks(SParams &P, unsigned int &grid1, const void *logits, const float *temp,
                 float2 *rec, WsHeader *hdr, int32_t R, int32_t V, int32_t dtype)
{
    const Layout lay = layout(R, V, dtype);
    const size_t NG = (lay.NS + GROUP - 1) / GROUP;
    const size_t groups = (size_t)R * NG;
    if ((size_t)R * lay.NS >= 0x7fffffffull)
        return SPEC_EINVAL;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SPEC_ECUDA;
    DevCache &dc = g_dev[dev];
    const int di = (dtype == SPEC_F32) ? 0 : 1;
    const void *fn = (dtype == SPEC_F32) ? (const void *)chunk_kernel<SPEC_F32>
                                         : (const void *)chunk_kernel<SPEC_BF16>;
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
    const size_t resident = (size_t)dc.sms.load(std::memory_order_relaxed) *
                            (size_t)dc.ctas_per_sm[di].load(std::memory_order_relaxed);
    grid1 = (unsigned int)(groups < resident ? groups : resident);

    P.logits = logits;
    P.u = nullptr;
    P.temperature = temp;
    P.out = nullptr;
    P.hdr = hdr;
    P.rec = rec;
    P.R = R;
    P.V = V;
    P.NS = (int)lay.NS;
    P.NC = (int)lay.NC;
    P.NG = (int)NG;
    P.total_groups = (unsigned int)groups;
    P.bytes = (unsigned long long)R * (unsigned long long)V * ((dtype == SPEC_F32) ? 4 : 2);
    P.rows_per_temp = 1;
    P.skip_greedy = 0;
    P.rjob = nullptr;
    P.rkcnt = nullptr;
    P.guard = 0.0f;
    return SPEC_OK;
}

// The fp32 draw's guard: a draw whose u * R lies within this fraction of R
// of the chosen cell's edges is drawn again exactly.  The fp32 record sums
// err by under 3e-7 of R (measured against the fp64 oracle over ~2100 bonus
// draws of the synthetic workloads, the same record search); the guard
// leaves a factor of 4.
constexpr float SAMPLE_GUARD = 1.2e-6f;

int launch(const void *logits, const float *u, const float *temp, int32_t *out, int32_t R,
           int32_t V, int32_t dtype, void *ws, size_t ws_size, void *stream,
           void *const *events)
{
    if (!sizes_ok(R, V, dtype))
        return SPEC_EINVAL;
    if (R == 0)
        return SPEC_OK;
    if (!logits || !u || !temp || !out || !ws)
        return SPEC_EINVAL;
    if ((reinterpret_cast<uintptr_t>(logits) & 15) || (reinterpret_cast<uintptr_t>(ws) & 15) ||
        (reinterpret_cast<uintptr_t>(u) & 3) || (reinterpret_cast<uintptr_t>(temp) & 3) ||
        (reinterpret_cast<uintptr_t>(out) & 3))
        return SPEC_EINVAL;
    const Layout lay = layout(R, V, dtype);
    if (ws_size < lay.total)
        return SPEC_ENOSPACE;
    uint8_t *w = reinterpret_cast<uint8_t *>(ws);
    SParams P;
    unsigned int grid1 = 0;
    const int rc = setup_chunks(P, grid1, logits, temp, reinterpret_cast<float2 *>(w + lay.rec),
                                reinterpret_cast<WsHeader *>(w), R, V, dtype);
    if (rc != SPEC_OK)
        return rc;
    P.u = u;
    P.out = out;
    RParams RP;
    resolve_regions(RP, w + lay.resolve, (size_t)R, V, false);
    RP.hdr = P.hdr;
    RP.out = out;
    RP.out_draw = nullptr;
    RP.rkink = nullptr;
    P.rjob = const_cast<RJob *>(RP.rjob);
    P.rkcnt = RP.rkcnt;
    P.guard = SAMPLE_GUARD;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SPEC_ECUDA;
    const size_t n_sms = (size_t)g_dev[dev].sms.load(std::memory_order_relaxed);  // set by setup_chunks
    const size_t ritems = (size_t)R * (size_t)RP.RNC;
    const unsigned int gridr = (unsigned int)(ritems < 3 * n_sms ? ritems : 3 * n_sms);
    const unsigned int gridrf = (unsigned int)((size_t)R < n_sms ? (size_t)R : n_sms);

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return (dtype == SPEC_F32) ? launch_all<SPEC_F32>(P, RP, gridr, gridrf, grid1, st, events)
                               : launch_all<SPEC_BF16>(P, RP, gridr, gridrf, grid1, st, events);
}

// host arena: logits | u | temperature | out | workspace, each 256-byte aligned
struct HostArena {
    size_t logits, u, temp, out, ws, total;
};

HostArena host_arena(int32_t R, int32_t V, int32_t dtype)
{
    HostArena h;
    const size_t es = (dtype == SPEC_F32) ? 4 : 2;
    h.logits = 0;
    h.u = align_up((size_t)R * V * es, 256);
    h.temp = h.u + align_up((size_t)R * 4, 256);
    h.out = h.temp + align_up((size_t)R * 4, 256);
    h.ws = h.out + align_up((size_t)R * 4, 256);
    h.total = h.ws + layout(R, V, dtype).total;
    return h;
}

}  // namespace

namespace spec_internal {

size_t chunk_count(int32_t V, int32_t dtype)
{
    return layout(1, V, dtype).NC;
}

int chunk_records(const void *logits, const float *temperature, int32_t rows_per_temp,
                  float2 *rec, void *hdr, int32_t R, int32_t V, int32_t dtype,
                  cudaStream_t stream)
{
    if (!sizes_ok(R, V, dtype) || rows_per_temp < 1)
        return SPEC_EINVAL;
    if (R == 0)
        return SPEC_OK;
    SParams P;
    unsigned int grid1 = 0;
    const int rc = setup_chunks(P, grid1, logits, temperature, rec,
                                reinterpret_cast<WsHeader *>(hdr), R, V, dtype);
    if (rc != SPEC_OK)
        return rc;
    P.rows_per_temp = rows_per_temp;
    P.skip_greedy = 1;
    if (dtype == SPEC_F32)
        chunk_kernel<SPEC_F32><<<grid1, NTHREADS, SMEM_BYTES, stream>>>(P);
    else
        chunk_kernel<SPEC_BF16><<<grid1, NTHREADS, SMEM_BYTES, stream>>>(P);
    if (cudaPeekAtLastError() != cudaSuccess) {
        (void)cudaGetLastError();
        return SPEC_ECUDA;
    }
    return SPEC_OK;
}

}  // namespace spec_internal

// ------------------------------------------------------------------- C ABI

extern "C" {

size_t spec_sample_workspace_size(int32_t R, int32_t V, int32_t dtype)
{
    if (!sizes_ok(R, V, dtype))
        return 0;
    return layout(R, V, dtype).total;
}

int32_t spec_sample(const void *logits, const float *u, const float *temperature,
                    int32_t *out_tokens, int32_t R, int32_t V, int32_t dtype,
                    void *workspace, size_t workspace_bytes, void *stream)
{
    return launch(logits, u, temperature, out_tokens, R, V, dtype, workspace, workspace_bytes,
                  stream, nullptr);
}

int32_t spec_sample_timed(const void *logits, const float *u, const float *temperature,
                          int32_t *out_tokens, int32_t R, int32_t V, int32_t dtype,
                          void *workspace, size_t workspace_bytes, void *stream,
                          void *const *stage_events)
{
    return launch(logits, u, temperature, out_tokens, R, V, dtype, workspace, workspace_bytes,
                  stream, stage_events);
}

size_t spec_sample_host_arena_size(int32_t R, int32_t V, int32_t dtype)
{
    if (!sizes_ok(R, V, dtype))
        return 0;
    return host_arena(R, V, dtype).total;
}

int32_t spec_sample_host(const void *logits, const float *u, const float *temperature,
                         int32_t *out_tokens, int32_t R, int32_t V, int32_t dtype,
                         void *device_arena, size_t arena_bytes, void *stream)
{
    if (!sizes_ok(R, V, dtype))
        return SPEC_EINVAL;
    if (R == 0)
        return SPEC_OK;
    if (!logits || !u || !temperature || !out_tokens || !device_arena)
        return SPEC_EINVAL;
    if (reinterpret_cast<uintptr_t>(device_arena) & 255)
        return SPEC_EINVAL;
    const HostArena h = host_arena(R, V, dtype);
    if (arena_bytes < h.total)
        return SPEC_ENOSPACE;
    const size_t es = (dtype == SPEC_F32) ? 4 : 2;
    uint8_t *a = reinterpret_cast<uint8_t *>(device_arena);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(a + h.logits, logits, (size_t)R * V * es, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaMemcpyAsync(a + h.u, u, (size_t)R * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(a + h.temp, temperature, (size_t)R * 4, cudaMemcpyHostToDevice, st) !=
            cudaSuccess)
        return SPEC_ECUDA;
    if (cudaMemsetAsync(a + h.ws, 0, sizeof(WsHeader), st) != cudaSuccess)
        return SPEC_ECUDA;
    const int rc = launch(a + h.logits, reinterpret_cast<const float *>(a + h.u),
                          reinterpret_cast<const float *>(a + h.temp),
                          reinterpret_cast<int32_t *>(a + h.out), R, V, dtype, a + h.ws,
                          h.total - h.ws, stream, nullptr);
    if (rc != SPEC_OK)
        return rc;
    if (cudaMemcpyAsync(out_tokens, a + h.out, (size_t)R * 4, cudaMemcpyDeviceToHost, st) !=
        cudaSuccess)
        return SPEC_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return SPEC_ECUDA;
    return SPEC_OK;
}

}  // extern "C"
