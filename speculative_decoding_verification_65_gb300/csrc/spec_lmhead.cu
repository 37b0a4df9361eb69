// spec_lmhead.cu -- verification with the target's LM head fused in: the
// target logits t = h W^T are computed tile by tile on the tcgen05 tensor
// cores and reduced to row statistics in the GEMM epilogue, so they never
// reach HBM.  C ABI in include/spec_lmhead.h.
//
// The pages place the verification right after one target forward pass that
// scores all k+1 positions ("Speculative Decoding and the Art of Fast LLM
// Inference", "The Algorithm, Step by Step", the verify step); the last layer
// of that pass is the LM head.  Fusing it changes where t comes from, not
// what the verification computes: accept test, first rejection, correction
// or bonus draw are those of spec_verify (include/spec_verify.h).
//
// Stages, in order on the caller's stream:
//   1. draft chunk records (the sampler's chunk kernel over the B*k draft rows)
//   2. gemm<STATS>: per (row, 256-column tile) (max, sum 2^((t-max)c), argmax),
//      and t(g) for the rows whose draft token falls in the tile
//   3. scan: fold the records, accept tests, first rejection; the draw row's
//      hidden vector is copied to a compact [B, d] buffer
//   4. gemm<DRAW>: the draw rows' logits again, reduced to the weight sum of
//      each 32-token group (residual max(0, p - q), or p for the bonus row)
//   5. final: inverse CDF over the group sums, the crossing group's 32 logits
//      recomputed as dot products, the token located in it
//
// Design of the GEMM (tcgen05, one CTA per SM, persistent):
//   - tile 128 rows x 256 columns, fp32 accumulator in tensor memory (TMEM),
//     two accumulators (512 columns) so the epilogue of one tile overlaps
//     the MMAs of the next
//   - warp 0: TMA producer (cp.async.bulk.tensor, 128-byte swizzle), a ring
//     of STAGES stages of 64 K-elements (16 KB of h, 32 KB of W)
//   - warp 1: TMEM allocation, and one thread issuing tcgen05.mma (M=128,
//     N=256, K=16, bf16 in, fp32 accumulate), committing to mbarriers
//   - warps 2..: the epilogue, one TMEM lane (one row) per thread; in the
//     draw GEMM two warps share a lane quarter, one half of the columns each
//   - tiles are ordered column-block major, so the CTAs working at one time
//     share a few 2 MB W tiles in L2 and W is read from HBM about once
// Every mbarrier wait is bounded; a wait that gives up sets
// SPEC_DEV_WAIT_TIMEOUT, the CTA stops issuing, lets its copies and MMAs in
// flight land (bounded again), frees its TMEM and returns.

#include <cuda.h>
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "spec_lmhead.h"
#include "internal.h"
#include "device_common.cuh"

using namespace spec_dev;

namespace {

constexpr int BM = 128;                   // rows per tile (TMEM lanes)
constexpr int BN = 256;                   // vocabulary columns per tile
constexpr int BK = 64;                    // K elements per stage: one 128-byte row
constexpr int UK = 16;                    // K per tcgen05.mma, kind::f16
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BYTES = BN * BK * 2;      // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NACC = 2;                   // accumulators in TMEM
constexpr int TMEM_COLS = NACC * BN;      // 512: all of TMEM

constexpr int GROUP = 32;                 // tokens per draw record

enum { MODE_STORE = 0, MODE_STATS = 1, MODE_DRAW_F32 = 2, MODE_DRAW_BF16 = 3 };

// Epilogue warps: the statistics epilogue (one exponential per logit) keeps
// up with the MMAs with one warp per TMEM lane quarter; the draw epilogue
// (two exponentials and a draft read per logit) needs two per quarter, each
// taking one half of the tile's columns.
template <int MODE>
__host__ __device__ constexpr int epi_warps() { return (MODE == MODE_DRAW_F32 || MODE == MODE_DRAW_BF16) ? 8 : 4; }
template <int MODE>
__host__ __device__ constexpr int gthreads() { return (2 + epi_warps<MODE>()) * 32; }  // + TMA warp, MMA warp

struct GSmemTail {
    unsigned long long full[STAGES];
    unsigned long long empty[STAGES];
    unsigned long long acc_full[NACC];
    unsigned long long acc_empty[NACC];
    unsigned long long drain;
    uint32_t tmem_base;
    int abort_flag;
};
// stages (1024-byte aligned for the swizzle) + tail + slack for the alignment
constexpr size_t GSMEM_BYTES = (size_t)STAGES * STAGE_BYTES + sizeof(GSmemTail) + 1024;

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            unsigned long long *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
           "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both K-major bf16, fp32 accumulate
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on `bar` once every tcgen05.mma this thread issued before has completed
__device__ __forceinline__ void mma_commit(unsigned long long *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        :: "r"(smem_addr(bar)) : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes, one lane per thread
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    __syncwarp();  // .sync.aligned: the whole warp, converged
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major bf16 operand staged by TMA
// with the 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes
// apart (stride byte offset), descriptor version 1, swizzle mode 2 (128 B).
// The leading byte offset is unused for this layout (set to 16 bytes).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B bf16, both
// K-major, N = BN, M = BM.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

}  // namespace

namespace {

// Per draw row: what its weights are (scan -> gemm<DRAW> -> final).
struct DrawJob {
    int mode;         // JOB_NONE, JOB_RESIDUAL (w = max(0, p - q)), JOB_BONUS (w = p)
    int b, j;         // sequence, position of the draw row
    float mt, rzt;    // target row max and 1 / Z_t
    float md, rzd;    // draft row max and 1 / Z_d (residual)
    float c;          // log2(e) / T
    float u;          // the sequence's u_resample
};
enum { JOB_NONE = 0, JOB_RESIDUAL = 1, JOB_BONUS = 2 };

struct GParams {
    int M, N, Kd;            // rows, vocabulary (columns), hidden size
    int mt, nt, kbs;         // tiles along M and N; K stages per tile
    int total;               // mt * nt
    int *status;             // the workspace status word
    // MODE_STORE
    float *out;              // [M][N]
    // MODE_STATS
    float4 *part;            // [M][nt]: (max, sum 2^((t-max)c), argmax index bits, 0)
    float *tg;               // [M]: t(g) of the row's draft token (rows i < k)
    const int32_t *tokens;   // [B][k]
    const float *temperature;
    int k;                   // rows per sequence are k + 1
    // MODE_DRAW_F32 / MODE_DRAW_BF16
    const DrawJob *jobs;     // [M] (one row per sequence)
    float *grp;              // [M][ng]: weight sum of each GROUP-token group
    float *grp_p;            // [M][ng]: the same for p alone (residual rows: the
                             // fallback when rounding leaves no residual mass)
    int ng;
    const void *draft;       // [B][k][N] draft logits
    int draft_dtype;
};

__device__ __forceinline__ float draft_at(const GParams &P, size_t idx)
{
    if (P.draft_dtype == SPEC_F32)
        return __ldg(reinterpret_cast<const float *>(P.draft) + idx);
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(P.draft) + idx);
    return __uint_as_float((uint32_t)h << 16);
}

// v[o] for a run-time o in [0, 32), by a tree of selects on o's bits (an
// indexed read would put v in local memory)
__device__ __forceinline__ float pick32(const float (&v)[32], int o)
{
    float a[16], b[8], c[4], d[2];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        a[i] = (o & 16) ? v[i + 16] : v[i];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        b[i] = (o & 8) ? a[i + 8] : a[i];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        c[i] = (o & 4) ? b[i + 4] : b[i];
#pragma unroll
    for (int i = 0; i < 2; ++i)
        d[i] = (o & 2) ? c[i + 2] : c[i];
    return (o & 1) ? d[1] : d[0];
}

// The epilogue of one thread's share of a tile: row `row` of the tile's 128,
// the COLS accumulator columns of part h (h * COLS on) at TMEM address taddr.
template <int MODE>
__device__ __forceinline__ void epilogue(const GParams &P, uint32_t taddr, int row, int n, int h)
{
    constexpr int COLS = BN / (epi_warps<MODE>() / 4);
    const int col_base = n * BN + h * COLS;
    if (MODE == MODE_STORE) {
#pragma unroll 1
        for (int ch = 0; ch < COLS / 32; ++ch) {
            float v[32];
            tmem_ld32(taddr + (uint32_t)(ch * 32), v);
            if (row < P.M) {
                float *o = P.out + (size_t)row * P.N;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int col = col_base + ch * 32 + j;
                    if (col < P.N)
                        o[col] = v[j];
                }
            }
        }
    } else if (MODE == MODE_STATS) {
        const bool inrow = row < P.M;
        const int b = inrow ? row / (P.k + 1) : 0;
        const int i = inrow ? row - b * (P.k + 1) : 0;
        const float T = inrow ? __ldg(P.temperature + b) : 0.0f;
        const bool sample = inrow && temperature_valid(T) && T > 0.0f;
        const float c = sample ? LOG2E / T : 0.0f;
        const int g = (inrow && i < P.k) ? __ldg(P.tokens + (size_t)b * P.k + i) : -1;
        float mx = -INFINITY, s = 0.0f, tgv = 0.0f;
        int idx = INT_MAX;
        bool has_tg = false;
#pragma unroll 1
        for (int ch = 0; ch < COLS / 32; ++ch) {
            float v[32];
            tmem_ld32(taddr + (uint32_t)(ch * 32), v);
            const int col0 = col_base + ch * 32;
            float cm = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (col0 + j >= P.N)
                    v[j] = -INFINITY;  // past the vocabulary (the W rows TMA filled with 0)
                cm = fmax_nan(cm, v[j]);
            }
            int ci = INT_MAX;
#pragma unroll
            for (int j = 31; j >= 0; --j)
                if (v[j] == cm)
                    ci = j;  // lowest column attaining the chunk maximum
            const float mn = fmax_nan(mx, cm);
            if (cm > mx)
                idx = col0 + ci;  // an equal maximum keeps the earlier (lower) column
            if (sample && mn != -INFINITY) {
                float cs = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    cs += ex2((v[j] - mn) * c);
                s = rescale(s, mx, mn, c) + cs;
            }
            mx = mn;
            if (g >= col0 && g < col0 + 32) {
                tgv = pick32(v, g - col0);
                has_tg = true;
            }
        }
        if (inrow) {
            P.part[(size_t)row * P.nt + n] = make_float4(mx, s, __int_as_float(idx), 0.0f);
            if (has_tg)
                P.tg[row] = tgv;
        }
    } else {  // MODE_DRAW_F32 / MODE_DRAW_BF16: the draft's element size is fixed
        constexpr int es = (MODE == MODE_DRAW_F32) ? 4 : 2;
        const bool inrow = row < P.M;
        DrawJob J;
        J.mode = JOB_NONE;
        if (inrow)
            J = P.jobs[row];
        const bool resid = J.mode == JOB_RESIDUAL;
        const size_t drow = resid ? ((size_t)J.b * P.k + J.j) * (size_t)P.N : 0;
        const uint8_t *dbase = reinterpret_cast<const uint8_t *>(P.draft) + drow * es;
        // 16-byte loads of the draft row where it is aligned and whole
        const bool vec = resid && ((reinterpret_cast<uintptr_t>(dbase) & 15) == 0);
        // the draft values of one 32-column chunk: 64 (bf16) or 128 (f32) bytes
        auto load_draft = [&](int col0, uint4 (&dv)[8]) {
            if (vec && col0 + 32 <= P.N) {
                const uint4 *src = reinterpret_cast<const uint4 *>(dbase + (size_t)col0 * es);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < 2 * es)
                        dv[q] = __ldcs(src + q);
            }
        };
        auto draft_val = [&](const uint4 (&dv)[8], int col0, int j) -> float {
            if (vec && col0 + 32 <= P.N) {
                const uint4 w4 = dv[(j * es) >> 4];
                const int e = ((j * es) & 15) >> 2;  // 32-bit word within the 16 bytes
                const uint32_t word = (e == 0) ? w4.x : (e == 1) ? w4.y : (e == 2) ? w4.z : w4.w;
                if (es == 4)
                    return __uint_as_float(word);
                return __uint_as_float((j & 1) ? (word & 0xffff0000u) : (word << 16));
            }
            return draft_at(P, drow + col0 + j);
        };
        uint4 dv[8], dn[8];
        if (resid)
            load_draft(col_base, dv);
#pragma unroll 1
        for (int ch = 0; ch < COLS / 32; ++ch) {
            const int col0 = col_base + ch * 32;
            if (resid && ch + 1 < COLS / 32)
                load_draft(col0 + 32, dn);  // one chunk ahead
            float v[32];
            tmem_ld32(taddr + (uint32_t)(ch * 32), v);
            if (J.mode != JOB_NONE && col0 < P.N) {
                float ws = 0.0f, ps = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int col = col0 + j;
                    if (col < P.N) {
                        const float p = ex2((v[j] - J.mt) * J.c) * J.rzt;
                        float w = p;
                        if (resid)
                            w = fmaxf(p - ex2((draft_val(dv, col0, j) - J.md) * J.c) * J.rzd,
                                      0.0f);
                        ws += w;
                        ps += p;
                    }
                }
                P.grp[(size_t)row * P.ng + col0 / GROUP] = ws;
                if (resid)
                    P.grp_p[(size_t)row * P.ng + col0 / GROUP] = ps;
            }
            if (resid) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    dv[q] = dn[q];
            }
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(gthreads<MODE>(), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const GParams P)
{
    extern __shared__ uint8_t gsm_raw[];
    const uint32_t raw = smem_addr(gsm_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;  // the swizzle wants 1024-byte stages
    const uint32_t sbase = raw + pad;
    GSmemTail &S = *reinterpret_cast<GSmemTail *>(gsm_raw + pad + (size_t)STAGES * STAGE_BYTES);
    volatile int *abort_flag = &S.abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(&S.acc_full[a], 1);
            mbar_init(&S.acc_empty[a], epi_warps<MODE>());
        }
        mbar_init(&S.drain, 1);
        S.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prefetch_map(&mapA);
        prefetch_map(&mapB);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&S.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = S.tmem_base;
    const int G = (int)gridDim.x;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0u, issued_phase = 0u;  // per stage: a load issued, its phase
            bool ok = true;
            for (int t = blockIdx.x; t < P.total && ok; t += G) {
                const int n = t / P.mt, m = t - n * P.mt;
                for (int kb = 0; kb < P.kbs; ++kb) {
                    if (*abort_flag || !mbar_wait(&S.empty[stage], phase ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + (uint32_t)(stage * STAGE_BYTES);
                    mbar_arrive_expect_tx(&S.full[stage], STAGE_BYTES);
                    tma_load_2d(sa, &mapA, kb * BK, m * BM, &S.full[stage]);
                    tma_load_2d(sa + A_BYTES, &mapB, kb * BK, n * BN, &S.full[stage]);
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                atomicExch(P.status, SPEC_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
                for (int s = 0; s < STAGES; ++s)  // the loads in flight land first (bounded)
                    if ((issued >> s) & 1u)
                        (void)mbar_wait(&S.full[s], (issued_phase >> s) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, issued = false;
            for (int t = blockIdx.x; t < P.total && ok; t += G) {
                if (*abort_flag || !mbar_wait(&S.acc_empty[acc], acc_phase ^ 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tbase + (uint32_t)(acc * BN);
                for (int kb = 0; kb < P.kbs; ++kb) {
                    if (*abort_flag || !mbar_wait(&S.full[stage], phase)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = sbase + (uint32_t)(stage * STAGE_BYTES);
                    const uint64_t ad = sw128_desc(sa), bd = sw128_desc(sa + A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / UK; ++kk)  // +32 bytes along K per step
                        mma_bf16(d, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), IDESC,
                                 (kb | kk) ? 1u : 0u);
                    issued = true;
                    mma_commit(&S.empty[stage]);  // the stage is free once these MMAs read it
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                mma_commit(&S.acc_full[acc]);  // the accumulator is complete
                if (++acc == NACC) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) {
                atomicExch(P.status, SPEC_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
                if (issued) {  // the MMAs in flight complete before TMEM is freed (bounded)
                    mma_commit(&S.drain);
                    (void)mbar_wait(&S.drain, 0u);
                }
            }
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;              // the TMEM lane quarter this warp may read
        const int h = (warp - 2) >> 2;       // its part of the columns (draw GEMM: a half)
        constexpr int COLS = BN / (epi_warps<MODE>() / 4);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < P.total; t += G) {
            const int n = t / P.mt, m = t - n * P.mt;
            int ok = 1;
            if (lane == 0)
                ok = (!*abort_flag && mbar_wait(&S.acc_full[acc], acc_phase)) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);  // the warp takes one path
            if (!ok) {
                if (lane == 0) {
                    atomicExch(P.status, SPEC_DEV_WAIT_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            const int row = m * BM + q * 32 + lane;
            epilogue<MODE>(P, tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + h * COLS),
                           row, n, h);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&S.acc_empty[acc]);
            if (++acc == NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, TMEM_COLS);
    }
    // This grid may have started while the kernel before it (the draft chunk
    // records) still ran; finishing only after that grid has finished lets
    // the next kernel's wait cover both.
    wait_previous_kernel();
}

}  // namespace

namespace {

constexpr int SCAN_WARPS = 4;
constexpr int MAX_CHUNKS = (SPEC_MAX_V / GROUP + 127) / 128;  // 256 for 2^20 tokens

struct VParams {
    int B, k, V, d;
    int nt;                   // statistics records (tiles) per target row
    int NC;                   // draft chunk records per row
    int ng;                   // draw groups per row
    int draft_dtype;
    const float4 *part;       // [B(k+1)][nt]
    const float *tg;          // [B(k+1)]
    const float2 *rec;        // [B k][NC]
    const void *draft;        // [B][k][V]
    const uint16_t *hidden;   // [B(k+1)][d] bf16
    uint16_t *hdraw;          // [B][d] bf16: each sequence's draw row
    DrawJob *jobs;            // [B]
    const float *grp;         // [B][ng]
    const float *grp_p;       // [B][ng]
    const uint16_t *lm_head;  // [V][d] bf16
    const int32_t *tokens;
    const float *u_accept, *u_resample, *temperature;
    int32_t *out_tokens, *out_num;
    float *out_probs;         // [B][k][2] or null
};

__device__ __forceinline__ float draft_logit(const VParams &P, size_t idx)
{
    if (P.draft_dtype == SPEC_F32)
        return __ldg(reinterpret_cast<const float *>(P.draft) + idx);
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(P.draft) + idx);
    return __uint_as_float((uint32_t)h << 16);
}

// (max, scaled sum, lowest argmax) of two row pieces
__device__ __forceinline__ void fold2(float &m, float &s, int &ix, float m2, float s2, int ix2,
                                      float c, bool sample)
{
    const float mn = fmax_nan(m, m2);
    if (sample)
        s = rescale(s, m, mn, c) + rescale(s2, m2, mn, c);
    ix = (m == mn && m2 == mn) ? min(ix, ix2) : ((m2 == mn) ? ix2 : ix);
    m = mn;
}

// Fold n pieces at stride 1 starting at `base` (float4: max, sum, index bits)
// across the warp; every lane returns the row's totals.
__device__ __forceinline__ void fold_row(const float4 *base, int n, float c, bool sample,
                                         int lane, float &m, float &s, int &ix)
{
    m = -INFINITY;
    s = 0.0f;
    ix = INT_MAX;
#pragma unroll 4
    for (int q = lane; q < n; q += 32) {
        const float4 v = __ldcg(base + q);
        fold2(m, s, ix, v.x, v.y, __float_as_int(v.z), c, sample);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, ix, o);
        fold2(m, s, ix, m2, s2, i2, c, sample);
    }
}

// the draft chunk records (max, sum) of one row, folded across the warp
__device__ __forceinline__ void fold_rec(const float2 *base, int n, float c, int lane, float &m,
                                         float &s)
{
    m = -INFINITY;
    s = 0.0f;
#pragma unroll 4
    for (int q = lane; q < n; q += 32) {
        const float2 v = __ldcg(base + q);
        const float mn = fmax_nan(m, v.x);
        s = rescale(s, m, mn, c) + rescale(v.y, v.x, mn, c);
        m = mn;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const float mn = fmax_nan(m, m2);
        s = rescale(s, m, mn, c) + rescale(s2, m2, mn, c);
        m = mn;
    }
}

__device__ __forceinline__ bool bad_max(float m)
{
    return isnan(m) || isinf(m);  // NaN / +inf in the row, or the row all -inf
}

// One warp per sequence: row statistics, accept tests, first rejection; the
// outputs of greedy and error sequences; the draw job and row of the others.
__global__ void __launch_bounds__(SCAN_WARPS * 32) scan_kernel(const VParams P)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * SCAN_WARPS + warp;
    if (b >= P.B)
        return;
    const int k = P.k, V = P.V;
    const float T = __ldg(P.temperature + b);
    const int g = (lane < k) ? __ldg(P.tokens + (size_t)b * k + lane) : 0;
    const float ua = (lane < k) ? __ldg(P.u_accept + (size_t)b * k + lane) : 0.0f;
    const float ur = __ldg(P.u_resample + b);
    allow_next_kernel();
    wait_previous_kernel();  // the records come from the kernels before
    const bool tvalid = temperature_valid(T);
    const bool greedy = tvalid && T == 0.0f;
    const bool sample = tvalid && !greedy;
    const float c = sample ? LOG2E / T : 0.0f;
    bool err = !tvalid || __any_sync(0xffffffffu, lane < k && (g < 0 || g >= V));

    // target rows 0..k: lane r keeps row r's (max, sum, argmax)
    float tm = 0.0f, tz = 0.0f;
    int ta = 0;
    if (!err) {
        for (int r = 0; r <= k; ++r) {
            float m, s;
            int ix;
            fold_row(P.part + ((size_t)b * (k + 1) + r) * P.nt, P.nt, c, sample, lane, m, s, ix);
            err = err || bad_max(m);
            if (lane == r) {
                tm = m;
                tz = s;
                ta = ix;
            }
        }
    }
    DrawJob J;
    J.mode = JOB_NONE;
    J.b = b;
    J.j = 0;
    J.mt = J.rzt = J.md = J.rzd = J.c = 0.0f;
    J.u = ur;
    int j = 0;
    float Pv = NAN, Qv = NAN;
    if (!err && greedy) {
        const unsigned int mism = __ballot_sync(0xffffffffu, lane < k && g != ta);
        j = mism ? (__ffs(mism) - 1) : k;
        const int corr = __shfl_sync(0xffffffffu, ta, j);
        if (lane <= k)
            P.out_tokens[(size_t)b * (k + 1) + lane] = (lane < j) ? g : ((lane == j) ? corr : -1);
        if (lane == 0)
            P.out_num[b] = j;
    } else if (!err) {
        // draft rows 0..k-1: lane i keeps row i's (max, sum)
        float dm = 0.0f, dz = 0.0f;
        for (int i = 0; i < k; ++i) {
            float m, s;
            fold_rec(P.rec + ((size_t)b * k + i) * P.NC, P.NC, c, lane, m, s);
            err = err || bad_max(m);
            if (lane == i) {
                dm = m;
                dz = s;
            }
        }
        if (!err) {
            bool acc = true, bad = false;
            if (lane < k) {
                const float tgl = __ldcg(P.tg + (size_t)b * (k + 1) + lane);
                const float dg = draft_logit(P, ((size_t)b * k + lane) * (size_t)V + g);
                Pv = ex2((tgl - tm) * c) / tz;
                Qv = ex2((dg - dm) * c) / dz;
                bad = !(Qv > 0.0f);
                acc = !bad && (Pv >= Qv || ua < Pv / Qv);
            }
            const unsigned int stop = __ballot_sync(0xffffffffu, lane < k && (!acc || bad));
            j = stop ? (__ffs(stop) - 1) : k;
            const bool badj = __shfl_sync(0xffffffffu, bad, j & 31) && j < k;
            err = badj;
            if (!err) {
                J.mode = (j < k) ? JOB_RESIDUAL : JOB_BONUS;
                J.j = j;
                J.c = c;
                J.mt = __shfl_sync(0xffffffffu, tm, j);
                J.rzt = 1.0f / __shfl_sync(0xffffffffu, tz, j);
                J.md = __shfl_sync(0xffffffffu, dm, j & 31);
                J.rzd = 1.0f / __shfl_sync(0xffffffffu, dz, j & 31);
                if (lane <= k)
                    P.out_tokens[(size_t)b * (k + 1) + lane] = (lane < j) ? g : -1;
                if (lane == 0)
                    P.out_num[b] = j;
                // the draw row's hidden vector (d bf16, 16-byte pieces)
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    P.hidden + ((size_t)b * (k + 1) + j) * (size_t)P.d);
                uint4 *dst = reinterpret_cast<uint4 *>(P.hdraw + (size_t)b * P.d);
                for (int q = lane; q < P.d / 8; q += 32)
                    dst[q] = __ldg(src + q);
            }
        }
    }
    if (err) {
        if (lane <= k)
            P.out_tokens[(size_t)b * (k + 1) + lane] = -1;
        if (lane == 0)
            P.out_num[b] = -1;
        J.mode = JOB_NONE;
    }
    if (P.out_probs && lane < k) {
        P.out_probs[((size_t)b * k + lane) * 2] = (sample && !err) ? Pv : NAN;
        P.out_probs[((size_t)b * k + lane) * 2 + 1] = (sample && !err) ? Qv : NAN;
    }
    if (lane == 0)
        P.jobs[b] = J;
}

// One warp per sequence with a draw: the inverse CDF over the group sums in
// index order (each lane a contiguous range of groups, Kogge-Stone across
// lanes), then the crossing group's 32 logits recomputed as dot products and
// searched in order.
// The group's recomputed weights may differ from the GEMM's by rounding; a
// threshold they leave past the group's end takes its last positive weight.
__global__ void __launch_bounds__(SCAN_WARPS * 32) final_kernel(const VParams P)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * SCAN_WARPS + warp;
    allow_next_kernel();
    wait_previous_kernel();  // the group sums come from the draw GEMM
    if (b >= P.B)
        return;
    DrawJob J = P.jobs[b];
    if (J.mode == JOB_NONE)
        return;
    const int ng = P.ng;
    // The group sums are read as chunks of 128 (32 lanes x float4, coalesced):
    // chunk c holds groups 128c .. 128c+127 with lane l's float4 groups
    // 128c+4l .. 128c+4l+3, so lane order within a chunk is group order.
    // Totals: per chunk in shared memory, then the row's R = their sum in
    // chunk order; the crossing chunk, lane and group follow the same order.
    __shared__ float ctot[SCAN_WARPS][MAX_CHUNKS];
    const int nch = (ng + 127) / 128;
    auto group4 = [&](const float *a, int c) {
        const int g0 = c * 128 + lane * 4;
        if (g0 + 3 < ng && (ng & 3) == 0)
            return __ldcg(reinterpret_cast<const float4 *>(a + g0));
        float4 r = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (g0 < ng) r.x = __ldcg(a + g0);
        if (g0 + 1 < ng) r.y = __ldcg(a + g0 + 1);
        if (g0 + 2 < ng) r.z = __ldcg(a + g0 + 2);
        if (g0 + 3 < ng) r.w = __ldcg(a + g0 + 3);
        return r;
    };
    auto totals = [&](const float *a) {  // chunk totals; returns R
        float R = 0.0f;
#pragma unroll 4
        for (int c = 0; c < nch; ++c) {
            const float4 v = group4(a, c);
            float s4 = ((v.x + v.y) + v.z) + v.w;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                s4 += __shfl_xor_sync(0xffffffffu, s4, o);
            if (lane == 0)
                ctot[warp][c] = s4;
            R += s4;
        }
        __syncwarp();
        return R;
    };
    const float *w = P.grp + (size_t)b * ng;
    float tot = totals(w);
    if (J.mode == JOB_RESIDUAL && !(tot > 0.0f)) {
        // rounding left no residual mass: draw from p_j instead
        w = P.grp_p + (size_t)b * ng;
        J.mode = JOB_BONUS;
        tot = totals(w);
    }
    const float tau = J.u * tot;
    // the crossing chunk: the first whose running total passes tau
    int C = -1;
    float before = 0.0f;
    {
        float run = 0.0f;
        for (int c = 0; c < nch; ++c) {
            const float x = ctot[warp][c];
            if (run + x > tau) {
                C = c;
                break;
            }
            run += x;
        }
        if (C < 0) {  // rounding: the last chunk with positive weight
            run = 0.0f;
            float lastrun = 0.0f;
            for (int c = 0; c < nch; ++c) {
                const float x = ctot[warp][c];
                if (x > 0.0f) {
                    C = c;
                    lastrun = run;
                }
                run += x;
            }
            run = lastrun;
            if (C < 0)
                C = 0;
        }
        before = run;
    }
    // within the chunk: lanes in order, then the lane's four groups
    int G;
    {
        const float4 v = group4(w, C);
        const float s4 = ((v.x + v.y) + v.z) + v.w;
        float incl = s4;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        const unsigned int cross = __ballot_sync(0xffffffffu, before + incl > tau);
        const unsigned int posm = __ballot_sync(0xffffffffu, s4 > 0.0f);
        const int L = cross ? (__ffs(cross) - 1) : (posm ? (31 - __clz(posm)) : 0);
        float run = before + __shfl_sync(0xffffffffu, incl - s4, L);
        const float4 vl = make_float4(__shfl_sync(0xffffffffu, v.x, L),
                                      __shfl_sync(0xffffffffu, v.y, L),
                                      __shfl_sync(0xffffffffu, v.z, L),
                                      __shfl_sync(0xffffffffu, v.w, L));
        const float e4[4] = {vl.x, vl.y, vl.z, vl.w};
        int gi = -1, lastpos = -1;
        float runpos = run;
        for (int e = 0; e < 4; ++e) {
            if (e4[e] > 0.0f) {
                lastpos = e;
                runpos = run;
            }
            if (gi < 0 && run + e4[e] > tau) {
                gi = e;
                break;
            }
            run += e4[e];
        }
        if (gi < 0) {  // rounding inside the lane's groups: its last positive one
            gi = lastpos >= 0 ? lastpos : 0;
            run = runpos;
        }
        G = C * 128 + L * 4 + gi;
        before = run;
    }
    if (G >= ng)
        G = ng - 1;

    // the group's 32 logits again, t(x) = h . W[x]: the warp reads each of
    // the 32 rows of W coalesced (lane l takes the 16-byte pieces l, l+32, ...),
    // sums its products in order and the lanes' sums are added by a butterfly;
    // lane r keeps row r's logit
    const int x = G * GROUP + lane;
    float t = -INFINITY;
    {
        const uint4 *hv = reinterpret_cast<const uint4 *>(P.hdraw + (size_t)b * P.d);
        const int nq = P.d / 8;  // 16-byte pieces per row
        for (int r0 = 0; r0 < 32; r0 += 4) {
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int q = lane; q < nq; q += 32) {
                const uint4 h4 = __ldcg(hv + q);
                const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int xr = min(G * GROUP + r0 + r, P.V - 1);  // rows past V: unused
                    const uint4 w4 = __ldg(reinterpret_cast<const uint4 *>(
                                               P.lm_head + (size_t)xr * P.d) + q);
                    const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[r] = fmaf(__uint_as_float(hw[e] << 16),
                                      __uint_as_float(ww[e] << 16), acc[r]);
                        acc[r] = fmaf(__uint_as_float(hw[e] & 0xffff0000u),
                                      __uint_as_float(ww[e] & 0xffff0000u), acc[r]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
                if (lane == r0 + r && x < P.V)
                    t = acc[r];
            }
        }
    }
    float wx = 0.0f;
    if (x < P.V) {
        const float p = ex2((t - J.mt) * J.c) * J.rzt;
        wx = p;
        if (J.mode == JOB_RESIDUAL)
            wx = fmaxf(p - ex2((draft_logit(P, ((size_t)b * P.k + J.j) * (size_t)P.V + x) -
                                J.md) * J.c) * J.rzd, 0.0f);
    }
    float cw = wx;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, cw, o);
        if (lane >= o)
            cw += y;
    }
    const unsigned int hit = __ballot_sync(0xffffffffu, x < P.V && before + cw > tau && wx > 0.0f);
    int tok;
    if (hit) {
        tok = G * GROUP + (__ffs(hit) - 1);
    } else {
        const unsigned int pos = __ballot_sync(0xffffffffu, wx > 0.0f);
        tok = G * GROUP + (pos ? (31 - __clz(pos)) : 0);
    }
    if (lane == 0)
        P.out_tokens[(size_t)b * (P.k + 1) + J.j] = tok;
}

}  // namespace

// ---------------------------------------------------------------- host side

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (a function-local static:
// its initialisation is thread-safe).
EncodeTiledFn encode_fn()
{
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        (void)cudaGetLastError();
        return nullptr;
    }();
    return fn;
}

// A [rows, d] bf16 row-major matrix as TMA tiles of box_rows x 64 elements
// (128 bytes, the 128-byte swizzle); rows past the end read as zero.
bool make_map(CUtensorMap *map, const void *base, int rows, int d, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The GEMMs count tiles in int: keep M x V's tile count well inside it.
bool tiles_ok(size_t M, int32_t V)
{
    return ((M + BM - 1) / BM) * (((size_t)V + BN - 1) / BN) <= ((size_t)1 << 30);
}

bool sizes_ok(int32_t B, int32_t k, int32_t V, int32_t d, int32_t ddt)
{
    return B >= 1 && k >= 1 && k <= 31 && V >= 2 && V <= SPEC_MAX_V && d >= 64 && d <= 16384 &&
           d % 64 == 0 && (ddt == SPEC_F32 || ddt == SPEC_BF16) &&
           (size_t)B * (k + 1) <= 0x7fffffffull / 2 && tiles_ok((size_t)B * (k + 1), V);
}

struct Layout {
    size_t part, tg, rec, jobs, hdraw, grp, grp_p, total;
    int nt, NC, ng;
};

// header | part [M][nt] | tg [M] | draft records [B k][NC] | jobs [B] |
// draw rows [B][d] bf16 | group sums [B][ng] | p group sums [B][ng]
Layout layout(int32_t B, int32_t k, int32_t V, int32_t d, int32_t ddt)
{
    Layout w;
    const size_t M = (size_t)B * (k + 1);
    w.nt = (V + BN - 1) / BN;
    w.NC = (int)spec_internal::chunk_count(V, ddt);
    w.ng = (V + GROUP - 1) / GROUP;
    w.part = sizeof(WsHeader);
    w.tg = align_up(w.part + M * w.nt * sizeof(float4), 256);
    w.rec = align_up(w.tg + M * sizeof(float), 256);
    w.jobs = align_up(w.rec + (size_t)B * k * w.NC * sizeof(float2), 256);
    w.hdraw = align_up(w.jobs + (size_t)B * sizeof(DrawJob), 256);
    w.grp = align_up(w.hdraw + (size_t)B * d * 2, 256);
    w.grp_p = align_up(w.grp + (size_t)B * w.ng * sizeof(float), 256);
    w.total = align_up(w.grp_p + (size_t)B * w.ng * sizeof(float), 256);
    return w;
}

// Per-device launch facts, filled by the first call on each device; a flag
// is published with release order after what it guards (host threads may
// race here, repeating the same idempotent calls).
struct DevInfo {
    std::atomic<int> sms;
    std::atomic<bool> attr[4];
};
DevInfo g_dev[64];

template <int MODE>
int launch_gemm(const CUtensorMap &ma, const CUtensorMap &mb, GParams &P, int M, int N, int Kd,
                cudaStream_t st, bool early)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SPEC_ECUDA;
    DevInfo &di = g_dev[dev];
    int sms = di.sms.load(std::memory_order_relaxed);
    if (!sms) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms < 1)
            return SPEC_ECUDA;
        di.sms.store(sms, std::memory_order_relaxed);
    }
    if (!di.attr[MODE].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)GSMEM_BYTES) != cudaSuccess)
            return SPEC_ECUDA;
        di.attr[MODE].store(true, std::memory_order_release);
    }
    P.M = M;
    P.N = N;
    P.Kd = Kd;
    P.mt = (M + BM - 1) / BM;
    P.nt = (N + BN - 1) / BN;
    P.kbs = Kd / BK;
    P.total = P.mt * P.nt;
    const int grid = P.total < sms ? P.total : sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned int)grid);
    cfg.blockDim = dim3(gthreads<MODE>());
    cfg.dynamicSmemBytes = GSMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = early ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gemm_kernel<MODE>, ma, mb, P) != cudaSuccess) {
        (void)cudaGetLastError();
        return SPEC_ECUDA;
    }
    return SPEC_OK;
}

int launch_small(void (*fn)(const VParams), const VParams &V, int B, cudaStream_t st, bool early)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned int)((B + SCAN_WARPS - 1) / SCAN_WARPS));
    cfg.blockDim = dim3(SCAN_WARPS * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = early ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fn, V) != cudaSuccess) {
        (void)cudaGetLastError();
        return SPEC_ECUDA;
    }
    return SPEC_OK;
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool al4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

int verify_lmhead(const void *hidden, const void *lm_head, const void *draft,
                  const int32_t *tokens, const float *ua, const float *ur, const float *temp,
                  int32_t *out_tokens, int32_t *out_num, float *out_probs, int32_t B, int32_t k,
                  int32_t V, int32_t d, int32_t ddt, void *ws, size_t ws_bytes, void *stream,
                  void *const *events)
{
    if (!sizes_ok(B, k, V, d, ddt))
        return SPEC_EINVAL;
    if (!hidden || !lm_head || !draft || !tokens || !ua || !ur || !temp || !out_tokens ||
        !out_num || !ws)
        return SPEC_EINVAL;
    if (!al16(hidden) || !al16(lm_head) || !al16(draft) || !al16(ws) || !al4(tokens) ||
        !al4(ua) || !al4(ur) || !al4(temp) || !al4(out_tokens) || !al4(out_num) ||
        (out_probs && !al4(out_probs)))
        return SPEC_EINVAL;
    const Layout L = layout(B, k, V, d, ddt);
    if (ws_bytes < L.total)
        return SPEC_ENOSPACE;
    uint8_t *w = reinterpret_cast<uint8_t *>(ws);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int M = B * (k + 1);
    auto mark = [&](int i) {
        if (events && events[i])
            cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), st);
    };
    const bool early = events == nullptr;

    CUtensorMap mh, mw, md;
    uint16_t *hdraw = reinterpret_cast<uint16_t *>(w + L.hdraw);
    if (!make_map(&mh, hidden, M, d, BM) || !make_map(&mw, lm_head, V, d, BN) ||
        !make_map(&md, hdraw, B, d, BM))
        return SPEC_ECUDA;

    // 1. draft chunk records
    int rc = spec_internal::chunk_records(draft, temp, k, reinterpret_cast<float2 *>(w + L.rec),
                                          w, B * k, V, ddt, st);
    if (rc != SPEC_OK)
        return rc;
    mark(0);
    // 2. the target rows' statistics
    GParams G;
    memset(&G, 0, sizeof(G));
    G.status = reinterpret_cast<int *>(w);
    G.part = reinterpret_cast<float4 *>(w + L.part);
    G.tg = reinterpret_cast<float *>(w + L.tg);
    G.tokens = tokens;
    G.temperature = temp;
    G.k = k;
    rc = launch_gemm<MODE_STATS>(mh, mw, G, M, V, d, st, early);
    if (rc != SPEC_OK)
        return rc;
    mark(1);
    // 3. accept scan
    VParams Pv;
    Pv.B = B;
    Pv.k = k;
    Pv.V = V;
    Pv.d = d;
    Pv.nt = L.nt;
    Pv.NC = L.NC;
    Pv.ng = L.ng;
    Pv.draft_dtype = ddt;
    Pv.part = G.part;
    Pv.tg = G.tg;
    Pv.rec = reinterpret_cast<const float2 *>(w + L.rec);
    Pv.draft = draft;
    Pv.hidden = reinterpret_cast<const uint16_t *>(hidden);
    Pv.hdraw = hdraw;
    Pv.jobs = reinterpret_cast<DrawJob *>(w + L.jobs);
    Pv.grp = reinterpret_cast<const float *>(w + L.grp);
    Pv.grp_p = reinterpret_cast<const float *>(w + L.grp_p);
    Pv.lm_head = reinterpret_cast<const uint16_t *>(lm_head);
    Pv.tokens = tokens;
    Pv.u_accept = ua;
    Pv.u_resample = ur;
    Pv.temperature = temp;
    Pv.out_tokens = out_tokens;
    Pv.out_num = out_num;
    Pv.out_probs = out_probs;
    rc = launch_small(scan_kernel, Pv, B, st, early);
    if (rc != SPEC_OK)
        return rc;
    mark(2);
    // 4. the draw rows' group sums
    GParams Gd;
    memset(&Gd, 0, sizeof(Gd));
    Gd.status = G.status;
    Gd.jobs = Pv.jobs;
    Gd.grp = reinterpret_cast<float *>(w + L.grp);
    Gd.grp_p = reinterpret_cast<float *>(w + L.grp_p);
    Gd.ng = L.ng;
    Gd.k = k;
    Gd.draft = draft;
    Gd.draft_dtype = ddt;
    rc = (ddt == SPEC_F32) ? launch_gemm<MODE_DRAW_F32>(md, mw, Gd, B, V, d, st, false)
                           : launch_gemm<MODE_DRAW_BF16>(md, mw, Gd, B, V, d, st, false);
    if (rc != SPEC_OK)
        return rc;
    mark(3);
    // 5. final search
    rc = launch_small(final_kernel, Pv, B, st, early);
    if (rc != SPEC_OK)
        return rc;
    mark(4);
    if (cudaPeekAtLastError() != cudaSuccess) {
        (void)cudaGetLastError();
        return SPEC_ECUDA;
    }
    return SPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_verify_lmhead_workspace_size(int32_t B, int32_t k, int32_t V, int32_t d,
                                         int32_t draft_dtype)
{
    if (!sizes_ok(B, k, V, d, draft_dtype))
        return 0;
    return layout(B, k, V, d, draft_dtype).total;
}

int32_t spec_verify_lmhead(const void *hidden, const void *lm_head, const void *draft_logits,
                           const int32_t *draft_tokens, const float *u_accept,
                           const float *u_resample, const float *temperature,
                           int32_t *out_tokens, int32_t *out_num_accepted,
                           int32_t B, int32_t k, int32_t V, int32_t d, int32_t draft_dtype,
                           void *workspace, size_t workspace_bytes, void *stream)
{
    return verify_lmhead(hidden, lm_head, draft_logits, draft_tokens, u_accept, u_resample,
                         temperature, out_tokens, out_num_accepted, nullptr, B, k, V, d,
                         draft_dtype, workspace, workspace_bytes, stream, nullptr);
}

int32_t spec_verify_lmhead_timed(const void *hidden, const void *lm_head,
                                 const void *draft_logits, const int32_t *draft_tokens,
                                 const float *u_accept, const float *u_resample,
                                 const float *temperature, int32_t *out_tokens,
                                 int32_t *out_num_accepted, float *out_probs,
                                 int32_t B, int32_t k, int32_t V, int32_t d,
                                 int32_t draft_dtype, void *workspace, size_t workspace_bytes,
                                 void *stream, void *const *stage_events)
{
    return verify_lmhead(hidden, lm_head, draft_logits, draft_tokens, u_accept, u_resample,
                         temperature, out_tokens, out_num_accepted, out_probs, B, k, V, d,
                         draft_dtype, workspace, workspace_bytes, stream, stage_events);
}

int32_t spec_lmhead_logits(const void *hidden, const void *lm_head, float *out, int32_t M,
                           int32_t V, int32_t d, int32_t *status, void *stream)
{
    if (M < 1 || V < 2 || V > SPEC_MAX_V || d < 64 || d > 16384 || d % 64 != 0 ||
        !tiles_ok((size_t)M, V))
        return SPEC_EINVAL;
    if (!hidden || !lm_head || !out || !status || !al16(hidden) || !al16(lm_head) || !al4(out) ||
        !al4(status))
        return SPEC_EINVAL;
    CUtensorMap mh, mw;
    if (!make_map(&mh, hidden, M, d, BM) || !make_map(&mw, lm_head, V, d, BN))
        return SPEC_ECUDA;
    GParams G;
    memset(&G, 0, sizeof(G));
    G.status = status;
    G.out = out;
    return launch_gemm<MODE_STORE>(mh, mw, G, M, V, d, reinterpret_cast<cudaStream_t>(stream),
                                   false);
}

}  // extern "C"
