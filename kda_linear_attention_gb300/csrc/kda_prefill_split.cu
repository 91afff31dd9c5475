// Chunked KDA prefill in two tensor-core kernels: an intra-chunk kernel that
// runs on every (chunk, head) at once, and an inter-chunk state pass that
// walks each (sequence, head) through its chunks.
//
// Math (the recurrence of "Colibri Kimi K3 Metal backend", architecture
// section, unrolled over a chunk of L <= 64 tokens; b_r = sum_{t<=r} g_t):
//   G^qk_rs = sum_c q_rc k_sc e^{b_rc - b_sc} (s <= r),  G^kk likewise (s < r)
//   T  = (I + Diag(beta) G^kk)^-1 (unit lower triangular),  T' = (T - I) Diag(beta)
//   W  = T' K0 + Diag(beta) K0,        K0_r = e^{b_r} k_r
//   U  = T' V + Diag(beta) V - W S
//   O  = Q0 S + A' U + Diag(q_r.k_r) U,  Q0_r = e^{b_r} q_r,  A' = strictly lower G^qk
//   S <- Diag(e^{b_L}) S + Kbar^T U,      Kbar_s = e^{b_L - b_s} k_s
// Everything that does not involve the state S (the decay prefix sums, the
// two Gram matrices, the triangular solve for T, W, Q0, Kbar, A') depends on
// one chunk only; the intra-chunk kernel computes it for all chunks of all
// sequences in parallel and writes one record per (chunk, head).  The state
// pass then does, per chunk, two rounds of MMAs and two epilogues:
//   D_U[j][r] = -(W S)^T + (T' V)^T,   D_O[j][r] = (Q0 S)^T
//                                      (fp16 S, W, Q0; bf16 T', V)
//   u = D_U + beta v  (fp32; its fp16 copy in TMEM is round 2's operand)
//   D_O += (A' U)^T,   S^T += (Kbar^T U)^T                        (fp16)
// with S^T kept in fp32 in TMEM for the whole sequence (lane j, column i) and
// pre-scaled by e^{b_L} while the first round runs.
//
// Decay folding in the Gram matrices (16-row sub-blocks p, sigma_p = b at the
// last row of p): e^{b_r - b_s} = e^{b_r - sigma_p} e^{sigma_p - b_s}, the
// first factor in [1, e^75] and the second in (0, 1] for g >= -5; the query
// side is one operand X = [q e^{b - sigma} ; k e^{b - sigma}] (128 rows), the
// key side a stack of four operands k_s e^{sigma_p - b_s} (160 rows), and one
// M=128, N=160 MMA gives both Gram matrices.
//
// Precision: bf16 operands for the Gram matrices and T' (whose partner V
// arrives in bf16), with the diagonal blocks of the query-side Gram
// corrected by the keys' bf16 low parts; fp16 (11 significant bits) for
// every product with the state and its inputs: S's copy, W, Q0 and the W
// product's T Diag(beta) and K0 in round 1, A', Kbar and U in round 2.
// Each of those is bounded (|q|, |k| <= 1 after the L2 norm; the decay
// factors <= 1; S and u of the order of v), well inside fp16's range; u
// (and through it an overflowing state copy) is checked.  The diagonal
// terms (beta_r v_r, beta_r K0_r, (q_r.k_r) u_r) stay in fp32 outside the
// MMAs, and the state itself is fp32 in TMEM for the whole sequence.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "kda_internal.h"
#include "tc_layout.cuh"

namespace kda {

// Nonzero when a bounded wait in either kernel gave up, or the chunk plan
// did not fit the workspace.
__device__ unsigned int g_kda_device_error = 0;

namespace {
using namespace tc;

constexpr int C = 64;

// 1 / x on the hardware reciprocal (about 1 ulp; 1 / 0 = inf)
__device__ __forceinline__ float rcp_fast(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// min / max that return NaN when either operand is NaN
__device__ __forceinline__ float fmin_nan(float a, float b) {
    float r;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
// eight bf16 (one 16-byte chunk) <-> four channel pairs
__device__ __forceinline__ void unpack_bf8x2(uint4 u, float2 (&x)[4]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = __bfloat1622float2(h[e]);
}
__device__ __forceinline__ uint4 pack_bf8x2(const float2 (&x)[4]) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 hv = __floats2bfloat162_rn(x[e].x, x[e].y);
        w[e] = *reinterpret_cast<uint32_t *>(&hv);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void ld_f2x4(const float *p, float2 (&x)[4]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = make_float2(a.x, a.y); x[1] = make_float2(a.z, a.w);
    x[2] = make_float2(b.x, b.y); x[3] = make_float2(b.z, b.w);
}

// ---- the per-(chunk, head) record ------------------------------------------
// Each piece is stored in the shared-memory operand layout in which the state
// pass feeds it to the tensor cores, so that one bulk copy places it.  The
// intra-chunk kernel writes the pieces it stores from registers with
// streaming stores (st.global.cs): the state pass reads each record once.
constexpr uint32_t R_WQ = 0;        // [-W ; Q0] fp16, 128 rows x 128, K-major sw (two 16 KB halves)
constexpr uint32_t R_T = 32768;     // T' bf16, strictly lower 64 x 64 packed by K-step (tri_off), 5 KB
constexpr uint32_t R_A = 37888;     // A' fp16, the same packing, 5 KB
constexpr uint32_t R_KB = 43008;    // Kbar fp16 [s][i] sw (two 8 KB halves of 64 channels), 16 KB
constexpr uint32_t R_VEC = 59392;   // beta[64], q.k[64], e^{b_L}[128] (fp32)
constexpr uint32_t REC_BYTES = 60416;
static_assert(REC_BYTES % 1024 == 0 && R_KB % 1024 == 0, "records and their swizzled piece 1 KB aligned");

// The strictly lower triangular 64 x 64 tiles T' [r][s] and A' [r][s] are
// stored by K-step kk (columns s = 16 kk .. 16 kk + 15) with only the row
// groups that can be nonzero there, g = r / 8 >= 2 kk: block kk holds groups
// 2 kk .. 7, two 128-byte chunks each (8 rows x 8 columns, the interleaved
// K-major layout of the MMA operands: group stride 256 B, chunk stride
// 128 B), at tri_base(kk); 5120 bytes in all instead of 8192.  The state
// pass multiplies block kk with N = 64 - 16 kk into columns 16 kk ..
__host__ __device__ constexpr uint32_t tri_base(int kk) { return 256u * (uint32_t)(8 * kk - kk * (kk - 1)); }
constexpr uint32_t kTriBytes = tri_base(4);
static_assert(kTriBytes == 5120, "packed triangle size");
// element (r, s), for r / 8 >= 2 (s / 16) only
__device__ __forceinline__ uint32_t tri_off(int r, int s) {
    const int kk = s >> 4;
    return tri_base(kk) + (uint32_t)((r >> 3) - 2 * kk) * 256u + (uint32_t)((s >> 3) & 1) * 128u +
           (uint32_t)(r & 7) * 16u + (uint32_t)(s & 7) * 2u;
}

// ============================================================================
// chunk plan: chunk_off[n] = sum_{m<n} ceil(len_m / 64), chunk_off[N] = total,
// chunk_off[N + 1] = 0 (the counter from which the intra-chunk kernel's CTAs
// take jobs),
// and per global chunk gc its first token and row count, tab[gc] = (tok, Lc),
// so that the intra-chunk kernel finds a job's chunk with one 8-byte load.
// cu_seqlens must start at or above 0, never decrease and end at or below T
// (the call's precondition, which the host cannot read); otherwise the plan
// is emptied (every offset 0) and the device error word set, so that the
// intra-chunk kernel has no jobs and the state pass, finding the chunk
// counts inconsistent, skips every non-empty sequence: nothing is read or
// written past the buffers sized for T.
// ============================================================================
__global__ void __launch_bounds__(1024) chunk_plan_kernel(const int32_t *__restrict__ cu, int N, int T,
                                                          int32_t *__restrict__ chunk_off,
                                                          int2 *__restrict__ tab) {
    __shared__ int32_t s_scan[1024];
    __shared__ int32_t s_carry;
    __shared__ int s_bad;
    const int t = threadIdx.x;
    if (t == 0) {
        s_carry = 0;
        s_bad = (cu[0] < 0 || cu[N] > T) ? 1 : 0;
    }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + t;
        int v = 0;
        if (n < N) {
            if (cu[n + 1] < cu[n]) s_bad = 1;
            v = (max(cu[n + 1] - cu[n], 0) + C - 1) / C;
        }
        s_scan[t] = v;
        __syncthreads();
        for (int off = 1; off < 1024; off <<= 1) {
            const int x = t >= off ? s_scan[t - off] : 0;
            __syncthreads();
            s_scan[t] += x;
            __syncthreads();
        }
        const int carry = s_carry;
        if (n < N) chunk_off[n] = carry + s_scan[t] - v;
        __syncthreads();
        if (t == 1023) s_carry = carry + s_scan[1023];
        __syncthreads();
    }
    if (t == 0) {
        chunk_off[N] = s_bad ? 0 : s_carry;
        chunk_off[N + 1] = 0;              // the intra-chunk kernel's job counter
    }
    if (s_bad) {
        for (int n = t; n < N; n += 1024) chunk_off[n] = 0;
        if (t == 0) atomicOr(&g_kda_device_error, 1u);
        return;
    }
    __syncthreads();                       // chunk_off is complete (this block wrote it)
    const int total = s_carry;
    for (int gc = t; gc < total; gc += 1024) {
        int lo = 0, hi = N - 1;            // the sequence: the last n with chunk_off[n] <= gc
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (chunk_off[mid] <= gc) lo = mid;
            else hi = mid - 1;
        }
        const int tok = cu[lo] + (gc - chunk_off[lo]) * C;
        tab[gc] = make_int2(tok, min(C, cu[lo + 1] - tok));
    }
}

// ============================================================================
// intra-chunk kernel: persistent, two CTAs (256 threads each) per SM.  Job j
// is (chunk, head) = divmod(total - 1 - j, H) (last chunk first); CTA b
// takes jobs b and b + G (G = grid size), then further jobs from a counter,
// each two jobs ahead, and prefetches the next job's inputs while it
// finishes the current one: its q and k as soon as the Gram product has
// consumed X, its g (L2 prefetch early, shared memory once the W product is
// done).
// ============================================================================
constexpr int NTA = 256;
constexpr uint32_t SA_X = 0;              // 32 KB: q|k (TMA) -> X [128][128] sw (A of the Gram)
constexpr uint32_t SA_KH = 32768;         // 56 KB: g (TMA) -> Khat [160][128] and below it Klo
                                          //   [64][128], one [224][128] sw B operand of the Gram
constexpr uint32_t SA_M = SA_KH;          //   after the Gram: M / T fp32 [64][68] (17408 B)
constexpr uint32_t SA_Y = SA_KH + 17408;  //   solve temporaries (4 KB)
constexpr uint32_t SA_T = SA_KH + 24576;  //   T Diag(beta) fp16 il [r][s], rows 0..63 twice
                                          //   (16 KB: the M = 128 A operand of the W product)
constexpr uint32_t KH_HALF = 224 * 128;  // one 64-channel half of the Khat | Klo operand
constexpr uint32_t SA_K0 = 90112;         // 16 KB: K0 [64 s][128 i] fp16 sw (MN-major B of the W product)
constexpr uint32_t SA_MISC = 106496;
constexpr uint32_t MA_BETA = 0;           // float[64]
constexpr uint32_t MA_GAM = 256;          // float[128]  e^{b_L}
constexpr uint32_t MA_TAB = 768;          // int2[2]: chunk-table entries of the next two jobs
constexpr uint32_t MA_JOB = 784;          // int[2]: the next two jobs' indices
                                          // (792..1023 free)
constexpr uint32_t MA_TOT = 1024;         // float[4][128] sub-block totals, then carry - sigma_u,
                                          //   then the warps' q . k partials [8][64]
constexpr uint32_t MA_SIG = 3072;         // float[4][128] first-half scan totals, then e^{b_L - sigma_u}
constexpr uint32_t MA_DD = 5120;          // float[4][128] e^{sigma_0}, e^{sigma_w - sigma_{w-1}}
constexpr uint32_t MA_BAR = 7168;         // 3 x u64: q|k, g, MMA
constexpr uint32_t MA_TMEM = 7192;
constexpr uint32_t SMEM_A_USED = SA_MISC + 7200;
constexpr uint32_t SMEM_A_ALLOC = SMEM_A_USED + 1024;
static_assert(2 * (SMEM_A_ALLOC + 1024) <= 233472, "two intra-chunk CTAs per SM");
static_assert(SA_T + 16384 <= SA_K0 && SA_Y + 4096 <= SA_T, "solve space inside the Khat region");
static_assert(SA_KH + 2 * KH_HALF == SA_K0 && (SA_KH + KH_HALF) % 1024 == 0, "Khat | Klo operand");
static_assert(SA_Y + 32 * 40 * 4 <= SA_T, "the 32 x 32 solve temporary fits");
constexpr int MLD = 68;                   // row stride (floats) of M / T
constexpr int YLD = 40;                   // row stride (floats) of the 32x32 solve temporary
constexpr uint32_t TMA_G = 0;             // Gram D, 160 columns, then
constexpr uint32_t TMA_C = 160;           //   the correction of its diagonal q blocks, 64 columns
constexpr uint32_t TMA_W = 0;             // W, 128 columns (after the Gram epilogue)

struct Job {
    int h, gc, tok, Lc;
};

__global__ void __launch_bounds__(NTA, 2)
intra_chunk_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_g, const float *__restrict__ beta,
                   const int2 *__restrict__ tab, int32_t *__restrict__ chunk_off, int N,
                   int H, uint8_t *__restrict__ recs, int T, int max_chunks) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *s_beta = reinterpret_cast<float *>(sm + SA_MISC + MA_BETA);
    float *s_gam = reinterpret_cast<float *>(sm + SA_MISC + MA_GAM);
    float *s_tot = reinterpret_cast<float *>(sm + SA_MISC + MA_TOT);
    float *s_sig = reinterpret_cast<float *>(sm + SA_MISC + MA_SIG);
    float *s_dd = reinterpret_cast<float *>(sm + SA_MISC + MA_DD);
    float *s_el = s_sig;
    uint64_t *bar_qk = reinterpret_cast<uint64_t *>(sm + SA_MISC + MA_BAR);
    uint64_t *bar_g = bar_qk + 1;
    uint64_t *bar_mma = bar_qk + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + SA_MISC + MA_TMEM);

    const int t = threadIdx.x;
    const int warp = t >> 5;
    const int lane = t & 31;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;

    // job -> (head, global chunk, first token, rows); every thread decodes.
    // Jobs run from the last chunk down, so the records of the first chunks,
    // which the state pass reads first, are the most recently written and
    // still in L2 when it starts.
    const int total = chunk_off[N] * H;
    // A job's chunk-table entry is copied into shared memory (s_tab, slot
    // k & 1 for the CTA's k-th job) two jobs ahead, so that no decode waits
    // on a global load.
    int2 *s_tab = reinterpret_cast<int2 *>(sm + SA_MISC + MA_TAB);
    int *s_job = reinterpret_cast<int *>(sm + SA_MISC + MA_JOB);
    // Jobs: each CTA's first two are static (b and b + G); after that thread
    // 32 takes the job two ahead from a counter, so that CTAs that finish
    // early take more jobs and the grid ends together.
    const int G = (int)gridDim.x;
    auto take_job = [&]() -> int { return 2 * G + atomicAdd(chunk_off + N + 1, 1); };
    auto gc_of = [&](int job) -> int { return (total - 1 - job) / H; };
    auto prefetch_entry = [&](int job, int slot) {
        if (job < total) {
            cp_async8(s_tab + slot, tab + KDA_DBG_INDEX(g_kda_device_error, gc_of(job), 0, max_chunks));
            cp_async_commit();
        }
    };
    auto decode = [&](int job, int2 e) -> Job {
        Job J;
        const int jr = total - 1 - job;
        J.h = jr % H;
        J.gc = jr / H;
        J.tok = e.x;
        J.Lc = e.y;
        // debug builds: the job's record and tokens inside the buffers
        J.gc = KDA_DBG_INDEX(g_kda_device_error, J.gc, 0, max_chunks);
        J.tok = KDA_DBG_INDEX(g_kda_device_error, J.tok, 0, T);
        J.Lc = KDA_DBG_INDEX(g_kda_device_error, J.Lc, 1, T - J.tok + 1);
        return J;
    };
    // q and k land as the two 64-row halves of X (rows 0..63 q, 64..127 k)
    auto issue_qk = [&](const Job &J) {
        mbar_arrive_expect_tx(bar_qk, 32768);
        tma_load_3d(sm + SA_X, &map_q, bar_qk, 0, J.h, J.tok);
        tma_load_3d(sm + SA_X + 8192, &map_k, bar_qk, 0, J.h, J.tok);
        tma_load_3d(sm + SA_X + 16384, &map_q, bar_qk, 64, J.h, J.tok);
        tma_load_3d(sm + SA_X + 24576, &map_k, bar_qk, 64, J.h, J.tok);
    };
    auto issue_g = [&](const Job &J) {
        mbar_arrive_expect_tx(bar_g, 32768);
#pragma unroll
        for (int bx = 0; bx < 4; ++bx)
            tma_load_3d(sm + SA_KH + 8192 * bx, &map_g, bar_g, 32 * bx, J.h, J.tok);
    };
    auto load_beta = [&](const Job &J) -> float {
        return (t < J.Lc) ? beta[(size_t)(J.tok + t) * H + J.h] : 0.f;
    };

    int job = blockIdx.x;
    if (job >= total) return;
    Job J = decode(job, tab[KDA_DBG_INDEX(g_kda_device_error, gc_of(job), 0, max_chunks)]);
    if (t == 32) {                         // thread 32 takes every job and makes every table copy
        s_job[1] = job + G;
        prefetch_entry(job + G, 1);
    }
    if (warp == 0) tmem_alloc(s_tmem, 256);
    if (t == 0) {
        mbar_init(bar_qk, 1);
        mbar_init(bar_g, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        prefetch_tmap(&map_q);
        prefetch_tmap(&map_k);
        prefetch_tmap(&map_g);
        issue_qk(J);
        issue_g(J);
    }
    float bnext = (t < C) ? load_beta(J) : 0.f;
    sync_tc();
    const uint32_t tmem = *s_tmem;
    // Each job commits two MMA groups (the Gram: phase parity 0, W: parity 1)
    // and one phase on each load barrier (parity it & 1).  On a failed wait,
    // `fail_at` records what is still in flight: 1 = this job's loads, 2 = the
    // Gram, 3 = the W product and the next job's q and k.
    bool failed = false;
    int fail_at = 0, fail_it = 0;
    bool fail_next = false;

    for (int it = 0; !failed; ++it) {
    const int h = J.h, Lc = J.Lc;
    uint8_t *rec = recs + ((size_t)J.gc * H + h) * REC_BYTES;
    if (t < C) s_beta[t] = bnext;
    const int job_next = s_job[(it + 1) & 1];   // published by the barriers since it was taken
    const bool has_next = job_next < total;
    Job Jn = J;
    if (t == 32) cp_async_wait_all();  // the next job's table entry (published by the barrier)
    if (!wait_all(bar_qk, it & 1) || !wait_all(bar_g, it & 1)) { failed = true; fail_at = 1; fail_it = it; fail_next = has_next; break; }

    // the previous job's -W copy has left the K0 tile (published by the scan's barriers)
    if (t == 0) bulk_wait_read();
    {
        // ===== decay prefix sums: column scan in place in the g tile =========
        // thread = (channels 4qd..4qd+3, sub-block u); the tile is four 128B-
        // swizzled boxes of [64 rows][32 channels] fp32
        {
            // thread = (channels 4qd..4qd+3, sub-block u, 8-row half hf): local
            // prefix of its 8 rows; the second half then adds the first's total
            const int qd = t & 31, u = (t >> 5) & 3, hf = t >> 7;
            uint8_t *colp = sm + SA_KH + 8192 * (qd >> 3) + (16 * u + 8 * hf) * 128;
            float4 x[8];
#pragma unroll
            for (int rr = 0; rr < 8; ++rr)
                x[rr] = *reinterpret_cast<const float4 *>(colp + rr * 128 + (((qd & 7) ^ rr) << 4));
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            float glo = 0.f, ghi = 0.f;       // smallest and largest gate (NaN-propagating)
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                if (16 * u + 8 * hf + rr < Lc) {  // rows past the end add nothing
                    glo = fmin_nan(glo, fmin_nan(fmin_nan(x[rr].x, x[rr].y), fmin_nan(x[rr].z, x[rr].w)));
                    ghi = fmax_nan(ghi, fmax_nan(fmax_nan(x[rr].x, x[rr].y), fmax_nan(x[rr].z, x[rr].w)));
                    acc.x += x[rr].x; acc.y += x[rr].y; acc.z += x[rr].z; acc.w += x[rr].w;
                }
                x[rr] = acc;
            }
            // the decay folding below needs every gate in [-5, 0]: a gate
            // below that would overflow the folding factors, so it is reported
            // (as is a NaN, which fails both comparisons)
            const bool g_out = !(glo >= kGateMin && ghi <= 0.f);
            if (__any_sync(0xffffffffu, g_out) && lane == 0) atomicOr(&g_kda_device_error, kErrGateRange);
            float4 *half_tot = reinterpret_cast<float4 *>(s_sig) + u * 32 + qd;
            if (hf == 0) *half_tot = acc;
            __syncthreads();
            float4 base = make_float4(0.f, 0.f, 0.f, 0.f);
            if (hf == 1) base = *half_tot;
#pragma unroll
            for (int rr = 0; rr < 8; ++rr)
                *reinterpret_cast<float4 *>(colp + rr * 128 + (((qd & 7) ^ rr) << 4)) =
                    make_float4(x[rr].x + base.x, x[rr].y + base.y, x[rr].z + base.z, x[rr].w + base.w);
            // the sub-block total is also the prefix at its last valid row
            if (hf == 1)
                *reinterpret_cast<float4 *>(s_tot + u * 128 + 4 * qd) =
                    make_float4(acc.x + base.x, acc.y + base.y, acc.z + base.z, acc.w + base.w);
        }
        __syncthreads();
        if (t < 128) {
            const int lu = (Lc - 1) >> 4;
            float base[4], sg[4];
            float run = 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                base[u] = run;
                run += s_tot[u * 128 + t];
            }
            float bL = 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (u == lu) bL = base[u] + s_tot[u * 128 + t];
#pragma unroll
            for (int u = 0; u < 4; ++u) sg[u] = (u <= lu) ? base[u] + s_tot[u * 128 + t] : bL;
#pragma unroll
            for (int u = 0; u < 4; ++u) s_tot[u * 128 + t] = base[u] - sg[u];
            constexpr float kL2e = 1.4426950408889634f;    // e^x = 2^{x log2 e}
            const float d0 = ex2_approx(sg[0] * kL2e), d1 = ex2_approx((sg[1] - sg[0]) * kL2e),
                        d2 = ex2_approx((sg[2] - sg[1]) * kL2e), d3 = ex2_approx((sg[3] - sg[2]) * kL2e);
            s_dd[t] = d0;
            s_dd[128 + t] = d1;
            s_dd[256 + t] = d2;
            s_dd[384 + t] = d3;
            const float e1 = d0 * d1, e2 = e1 * d2, e3 = e2 * d3;
            const float l2 = d3, l1 = d2 * d3, l0 = d1 * l1;
            s_el[t] = l0;
            s_el[128 + t] = l1;
            s_el[256 + t] = l2;
            s_el[384 + t] = 1.f;
            s_gam[t] = e3;
        }
        __syncthreads();

        // ===== operand build: thread = row rb of every sub-block, channels 8cc..8cc+7
        const int rb = lane & 15;
        const int cc = 2 * warp + (lane >> 4);
        float F[4][8];                     // e^{b - sigma_u} (0 for rows past the end)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = 16 * u + rb;
            const bool valid = r < Lc;
            const uint8_t *rowp = sm + SA_KH + 8192 * (cc >> 2) + r * 128;
            const int c4 = 2 * (cc & 3);
            const float4 ga = *reinterpret_cast<const float4 *>(rowp + ((c4 ^ (r & 7)) << 4));
            const float4 gb = *reinterpret_cast<const float4 *>(rowp + (((c4 + 1) ^ (r & 7)) << 4));
            const float4 ba = *reinterpret_cast<const float4 *>(s_tot + u * 128 + 8 * cc);
            const float4 bb = *reinterpret_cast<const float4 *>(s_tot + u * 128 + 8 * cc + 4);
            // e^{b - sigma_u} = 2^{(b - sigma_u) log2 e}: the sums and their
            // scaling in packed pairs, the powers on the special-function unit
            const float2 l2e = make_float2(1.4426950408889634f, 1.4426950408889634f);
            const float2 gl[4] = {__fmul2_rn(__fadd2_rn(make_float2(ga.x, ga.y), make_float2(ba.x, ba.y)), l2e),
                                  __fmul2_rn(__fadd2_rn(make_float2(ga.z, ga.w), make_float2(ba.z, ba.w)), l2e),
                                  __fmul2_rn(__fadd2_rn(make_float2(gb.x, gb.y), make_float2(bb.x, bb.y)), l2e),
                                  __fmul2_rn(__fadd2_rn(make_float2(gb.z, gb.w), make_float2(bb.z, bb.w)), l2e)};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                F[u][2 * c] = valid ? ex2_approx(gl[c].x) : 0.f;
                F[u][2 * c + 1] = valid ? ex2_approx(gl[c].y) : 0.f;
            }
            // Q0 = q e^{b} -> record rows 64..127 of [-W ; Q0];  K0 = k e^{b} -> smem,
            // as (x e^{b - sigma}) e^{sigma}, while X still holds the raw rows
            // (here rather than in the operand build, whose live ranges are long)
            {
                float2 qv[4], kv[4], ep[4], q0[4], k0[4];
                unpack_bf8x2(*reinterpret_cast<const uint4 *>(sm + SA_X + sw_chunk(r, cc, 16384)), qv);
                unpack_bf8x2(*reinterpret_cast<const uint4 *>(sm + SA_X + sw_chunk(64 + r, cc, 16384)), kv);
                // e^{sigma_u} = e^{sigma_0} e^{sigma_1 - sigma_0} ...
                ld_f2x4(s_dd + 8 * cc, ep);
#pragma unroll
                for (int w = 1; w <= u; ++w) {
                    float2 dw[4];
                    ld_f2x4(s_dd + w * 128 + 8 * cc, dw);
#pragma unroll
                    for (int m = 0; m < 4; ++m) ep[m] = __fmul2_rn(ep[m], dw[m]);
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float2 F2 = make_float2(F[u][2 * m], F[u][2 * m + 1]);
                    q0[m] = __fmul2_rn(__fmul2_rn(qv[m], F2), ep[m]);
                    k0[m] = __fmul2_rn(__fmul2_rn(kv[m], F2), ep[m]);
                }
                __stcs(reinterpret_cast<uint4 *>(rec + R_WQ + sw_chunk(64 + r, cc, 16384)), pack_h8x2(q0));
                *reinterpret_cast<uint4 *>(sm + SA_K0 + sw_chunk(r, cc, 8192)) = pack_h8x2(k0);
            }
        }
        __syncthreads();                   // the g tile is read: Khat may be written

        float dqp[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = 16 * u + rb;
            uint8_t *pq = sm + SA_X + sw_chunk(r, cc, 16384);
            uint8_t *pk = sm + SA_X + sw_chunk(64 + r, cc, 16384);
            // channel pairs in packed fp32x2 arithmetic
            float2 qv[4], kv[4], F2[4], G2[4], xq[4], xk[4], el[4], kg[4];
            unpack_bf8x2(*reinterpret_cast<const uint4 *>(pq), qv);
            unpack_bf8x2(*reinterpret_cast<const uint4 *>(pk), kv);
            ld_f2x4(s_el + u * 128 + 8 * cc, el);
            float2 dot2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                F2[m] = make_float2(F[u][2 * m], F[u][2 * m + 1]);
                dot2 = __ffma2_rn(qv[m], kv[m], dot2);
                G2[m] = make_float2(F2[m].x > 0.f ? rcp_fast(F2[m].x) : 0.f,
                                    F2[m].y > 0.f ? rcp_fast(F2[m].y) : 0.f);
                xq[m] = __fmul2_rn(qv[m], F2[m]);
                xk[m] = __fmul2_rn(kv[m], F2[m]);
                kg[m] = __fmul2_rn(kv[m], G2[m]);
            }
            dqp[u] = (r < Lc) ? dot2.x + dot2.y : 0.f;
            // X in place: q rows 0..63, k rows 64..127
            *reinterpret_cast<uint4 *>(pq) = pack_bf8x2(xq);
            *reinterpret_cast<uint4 *>(pk) = pack_bf8x2(xk);
            // Khat stack: block pp >= u holds k_s e^{sigma_pp - b_s} at row 8pp(pp+1) + s
            float2 kh[4] = {kg[0], kg[1], kg[2], kg[3]};
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                if (pp >= u) {
                    if (pp > u) {
                        float2 dd[4];
                        ld_f2x4(s_dd + pp * 128 + 8 * cc, dd);
#pragma unroll
                        for (int m = 0; m < 4; ++m) kh[m] = __fmul2_rn(kh[m], dd[m]);
                    }
                    *reinterpret_cast<uint4 *>(sm + SA_KH + sw_chunk(8 * pp * (pp + 1) + r, cc, KH_HALF)) =
                        pack_bf8x2(kh);
                }
            }
            // the low part of the diagonal block's keys (block u of the stack
            // holds kg itself): lo(kg) = kg - bf16(kg), rounded to bf16, at row
            // 160 + r of the Gram's B operand (the correction columns)
            {
                float2 kl[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float2 kh2 = __bfloat1622float2(__floats2bfloat162_rn(kg[m].x, kg[m].y));
                    kl[m] = __ffma2_rn(kh2, make_float2(-1.f, -1.f), kg[m]);   // kg - kh2, exact product
                }
                *reinterpret_cast<uint4 *>(sm + SA_KH + sw_chunk(160 + r, cc, KH_HALF)) = pack_bf8x2(kl);
            }
            // Kbar = e^{b_L - b} k, fp16, row s, in the 128B-swizzled [s][i]
            // layout of K0: round 2 reads it as an MN-major operand
            {
                float2 kb[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) kb[m] = __fmul2_rn(kg[m], el[m]);
                __stcs(reinterpret_cast<uint4 *>(rec + R_KB + sw_chunk(r, cc, 8192)), pack_h8x2(kb));
            }
        }
        // q_r . k_r: each warp's partial over its 16 channels into the
        // sub-block totals' space (read before the block barrier above),
        // summed over the warps in a fixed order below, so that o is the same
        // bits on every call
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float d2 = dqp[u] + __shfl_xor_sync(0xffffffffu, dqp[u], 16);
            if (lane < 16) s_tot[warp * 64 + 16 * u + rb] = d2;
        }
        fence_proxy_async_smem();
        sync_tc();

        // ===== Gram: D[128 x 224] = X [Khat ; Klo]^T ========================
        // Columns 0..159 hold both gated Gram matrices; columns 160..223 the
        // diagonal q blocks of the Gram in more than bf16 precision, X Klo^T
        // (every q row against every diagonal key row; row r of sub-block p
        // uses columns 160 + 16p .. 160 + 16p + 15), added to hi(xq) hi(kg) in
        // the epilogue.  A' of a short sequence lives in these blocks, where
        // the bf16 rounding of the keys alone would cost o up to 2^-9 of each
        // product term.
        if (t == 0) {
            const uint32_t idg = instr_desc(kFmtBF16, 128, 224, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ko = (uint32_t)(kk >> 2), kb2 = (uint32_t)(kk & 3) * 32u;
                const uint64_t ax = smem_desc(smem_u32(sm + SA_X + ko * 16384 + kb2), 16, 1024, kSwizzle128B);
                const uint64_t bk = smem_desc(smem_u32(sm + SA_KH + ko * KH_HALF + kb2), 16, 1024, kSwizzle128B);
                mma_bf16_ss(tmem + TMA_G, ax, bk, idg, kk > 0);
            }
            mma_commit(bar_mma);
        }
        // while the Gram runs (thread 0 only issues it): the record's vectors
        // from warps 4..7, the next job's decode, its beta and an L2 pull of
        // its g from warps 0..3 and 1
        if (t >= 128) {
            const int i = t - 128;
            float *rv = reinterpret_cast<float *>(rec + R_VEC);
            if (i < 64) {
                float dq = s_tot[i];
#pragma unroll
                for (int w = 1; w < 8; ++w) dq += s_tot[w * 64 + i];
                rv[i] = s_beta[i];
                rv[64 + i] = dq;
            }
            rv[128 + i] = s_gam[i];
        }
        if (has_next) {
            Jn = decode(job_next, s_tab[(it + 1) & 1]);
            if (t == 32) {
                const int j2 = take_job();
                s_job[it & 1] = j2;
                prefetch_entry(j2, it & 1);
#pragma unroll
                for (int bx = 0; bx < 4; ++bx) tma_prefetch_l2_3d(&map_g, 32 * bx, Jn.h, Jn.tok);
            }
            if (t < C) bnext = load_beta(Jn);
        }
        if (!wait_all(bar_mma, 0)) { failed = true; fail_at = 2; fail_it = it; fail_next = has_next; break; }
    }
    {
        tc_fence_after();
        // X is consumed: the next job's q and k
        if (t == 0 && has_next) issue_qk(Jn);
        // ===== Gram epilogue -> A' (fp16, record) and M = Diag(beta) G^kk (fp32)
        float *Mm = reinterpret_cast<float *>(sm + SA_M);
        {
            const int ch = t & 127;
            const bool qside = ch < 64;
            const int r = ch & 63;
            const int p = r >> 4;
            const int plo = (r >> 5) * 2;
            const float br = s_beta[r];
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int qt = 2 * (t >> 7) + qq;
                const uint32_t col_lo = (uint32_t)min(8 * plo * (plo + 1) + 16 * qt, 144);
                const uint32_t col_hi = (uint32_t)min(8 * (plo + 1) * (plo + 2) + 16 * qt, 144);
                float va[16], vb[16], ca[16], cb[16];
                tmem_ld16(tmem + lane_base + TMA_G + col_lo, va);
                tmem_ld16(tmem + lane_base + TMA_G + col_hi, vb);
                if (qside) {                   // the diagonal correction of sub-blocks plo, plo + 1
                    tmem_ld16(tmem + lane_base + TMA_C + 16 * plo, ca);
                    tmem_ld16(tmem + lane_base + TMA_C + 16 * plo + 16, cb);
                }
                tmem_wait_ld();
                const bool use_hi = p != plo;
                const bool have = qt <= p && r < Lc;
                const bool diag = qside && qt == p;
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {   // 8 columns: one 16-byte chunk of the packing
                    float x8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = 16 * qt + 8 * jp + e;
                        float val = use_hi ? vb[8 * jp + e] : va[8 * jp + e];
                        if (diag) val += use_hi ? cb[8 * jp + e] : ca[8 * jp + e];
                        x8[e] = (have && s < r) ? val : 0.f;
                    }
                    if (qside) {
                        if ((r >> 3) >= 2 * qt)      // a row group that block qt of the packing holds
                            __stcs(reinterpret_cast<uint4 *>(rec + R_A + tri_off(r, 16 * qt + 8 * jp)),
                                   make_uint4(pack_h2(x8[0], x8[1]), pack_h2(x8[2], x8[3]),
                                              pack_h2(x8[4], x8[5]), pack_h2(x8[6], x8[7])));
                    } else {
                        float *mr = Mm + r * MLD + 16 * qt + 8 * jp;
                        *reinterpret_cast<float4 *>(mr) = make_float4(br * x8[0], br * x8[1], br * x8[2], br * x8[3]);
                        *reinterpret_cast<float4 *>(mr + 4) = make_float4(br * x8[4], br * x8[5], br * x8[6], br * x8[7]);
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();

        // ===== T = (I + M)^-1 by 16-row blocks, in place ======================
        float *Yt = reinterpret_cast<float *>(sm + SA_Y);
        {
            // diagonal blocks by forward substitution across a 16-lane group:
            // lane = row r, four right-hand sides (columns c0..c0+3) per thread
            const int r = t & 15;
            const int grp = t >> 4;
            const int p = grp >> 2, c0 = 4 * (grp & 3);
            float mr[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 m4 = *reinterpret_cast<const float4 *>(Mm + (16 * p + r) * MLD + 16 * p + 4 * j);
                mr[4 * j] = m4.x; mr[4 * j + 1] = m4.y; mr[4 * j + 2] = m4.z; mr[4 * j + 3] = m4.w;
            }
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = (r == c0 + e) ? 1.f : 0.f;
#pragma unroll
            for (int s2 = 0; s2 < 15; ++s2) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // rows r <= s2 have M[r][s2] = 0 (M is strictly lower), so
                    // every lane applies the update unconditionally
                    const float bv = __shfl_sync(0xffffffffu, x[e], s2, 16);
                    x[e] = fmaf(-mr[s2], bv, x[e]);
                }
            }
            __syncthreads();
            *reinterpret_cast<float4 *>(Mm + (16 * p + r) * MLD + 16 * p + c0) =
                make_float4(x[0], x[1], x[2], x[3]);
        }
        __syncthreads();
        // off-diagonal blocks, two levels: T_10 and T_32 (T_pq = -T_pp M_pq T_qq),
        // then the lower-left 32x32 block T_C = -T_B M_C T_A.  The 16x16
        // products run on warp-level tf32 MMAs in warps 0..3 (warp = block,
        // column tile of 8): P = M_pq T_qq into the temporary, then
        // T_pq = -T_pp P over M_pq
        {
            const int g = lane >> 2, tg = lane & 3;
            const int blk = (warp >> 1) & 1, nt = warp & 1;
            const int p = blk ? 3 : 1, q = p - 1;
            if (warp < 4) {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                for (int kk = nt; kk < 2; ++kk) {          // T_qq lower triangular
                    const float *A = Mm + (16 * p) * MLD + 16 * q + 8 * kk;
                    const float *Bm = Mm + (16 * q + 8 * kk) * MLD + 16 * q + 8 * nt;
                    const uint32_t a[4] = {to_tf32(A[g * MLD + tg]), to_tf32(A[(g + 8) * MLD + tg]),
                                           to_tf32(A[g * MLD + tg + 4]), to_tf32(A[(g + 8) * MLD + tg + 4])};
                    const uint32_t b[2] = {to_tf32(Bm[tg * MLD + g]), to_tf32(Bm[(tg + 4) * MLD + g])};
                    mma_tf32_16x8x8(d, a, b);
                }
                float *Y = Yt + (16 * blk) * 16 + 8 * nt;
                Y[g * 16 + 2 * tg] = d[0];
                Y[g * 16 + 2 * tg + 1] = d[1];
                Y[(g + 8) * 16 + 2 * tg] = d[2];
                Y[(g + 8) * 16 + 2 * tg + 1] = d[3];
            }
            __syncthreads();
            if (warp < 4) {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const float *A = Mm + (16 * p) * MLD + 16 * p + 8 * kk;
                    const float *Bm = Yt + (16 * blk + 8 * kk) * 16 + 8 * nt;
                    const uint32_t a[4] = {to_tf32(A[g * MLD + tg]), to_tf32(A[(g + 8) * MLD + tg]),
                                           to_tf32(A[g * MLD + tg + 4]), to_tf32(A[(g + 8) * MLD + tg + 4])};
                    const uint32_t b[2] = {to_tf32(Bm[tg * 16 + g]), to_tf32(Bm[(tg + 4) * 16 + g])};
                    mma_tf32_16x8x8(d, a, b);
                }
                float *Tq = Mm + (16 * p) * MLD + 16 * q + 8 * nt;
                Tq[g * MLD + 2 * tg] = -d[0];
                Tq[g * MLD + 2 * tg + 1] = -d[1];
                Tq[(g + 8) * MLD + 2 * tg] = -d[2];
                Tq[(g + 8) * MLD + 2 * tg + 1] = -d[3];
            }
        }
        __syncthreads();
        // lower-left 32x32 block on warp-level tf32 MMAs (8 warps: row tile mt,
        // column tile nt of 8); the triangular factors' zero tiles are skipped
        {
            // Y2 = M[32:64][0:32] T[0:32][0:32]   (T_A lower triangular: kk >= nt)
            const int g = lane >> 2, tg = lane & 3;
            const int mt = warp >> 2, nt = warp & 3;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            for (int kk = nt; kk < 4; ++kk) {
                const float *A = Mm + (32 + 16 * mt) * MLD + 8 * kk;
                const float *Bm = Mm + (8 * kk) * MLD + 8 * nt;
                const uint32_t a[4] = {to_tf32(A[g * MLD + tg]), to_tf32(A[(g + 8) * MLD + tg]),
                                       to_tf32(A[g * MLD + tg + 4]), to_tf32(A[(g + 8) * MLD + tg + 4])};
                const uint32_t b[2] = {to_tf32(Bm[tg * MLD + g]), to_tf32(Bm[(tg + 4) * MLD + g])};
                mma_tf32_16x8x8(d, a, b);
            }
            float *Y = Yt + (16 * mt) * YLD + 8 * nt;
            Y[g * YLD + 2 * tg] = d[0];
            Y[g * YLD + 2 * tg + 1] = d[1];
            Y[(g + 8) * YLD + 2 * tg] = d[2];
            Y[(g + 8) * YLD + 2 * tg + 1] = d[3];
        }
        __syncthreads();
        {
            // T_C = -T[32:64][32:64] Y2   (T_B lower triangular: kk <= 2 mt + 1)
            const int g = lane >> 2, tg = lane & 3;
            const int mt = warp >> 2, nt = warp & 3;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            for (int kk = 0; kk <= 2 * mt + 1; ++kk) {
                const float *A = Mm + (32 + 16 * mt) * MLD + 32 + 8 * kk;
                const float *Bm = Yt + (8 * kk) * YLD + 8 * nt;
                const uint32_t a[4] = {to_tf32(A[g * MLD + tg]), to_tf32(A[(g + 8) * MLD + tg]),
                                       to_tf32(A[g * MLD + tg + 4]), to_tf32(A[(g + 8) * MLD + tg + 4])};
                const uint32_t b[2] = {to_tf32(Bm[tg * YLD + g]), to_tf32(Bm[(tg + 4) * YLD + g])};
                mma_tf32_16x8x8(d, a, b);
            }
            float *Tc = Mm + (32 + 16 * mt) * MLD + 8 * nt;
            Tc[g * MLD + 2 * tg] = -d[0];
            Tc[g * MLD + 2 * tg + 1] = -d[1];
            Tc[(g + 8) * MLD + 2 * tg] = -d[2];
            Tc[(g + 8) * MLD + 2 * tg + 1] = -d[3];
        }
        __syncthreads();
        // T' = (T - I) Diag(beta), bf16 K-major il [r][s], to the record (B of
        // the U~ product in the state pass); T Diag(beta) = T' + Diag(beta) to
        // shared memory (A of the W product)
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            // a warp writes 8 rows x 4 chunks: whole 128-byte lines of the il layout
            const int r = 8 * warp + (lane & 7), s0 = 8 * ((lane >> 3) + 4 * pass);
            const float4 a = *reinterpret_cast<const float4 *>(Mm + r * MLD + s0);
            const float4 b4 = *reinterpret_cast<const float4 *>(Mm + r * MLD + s0 + 4);
            const float tv[8] = {a.x, a.y, a.z, a.w, b4.x, b4.y, b4.z, b4.w};
            const float4 ba = *reinterpret_cast<const float4 *>(s_beta + s0);
            const float4 bb = *reinterpret_cast<const float4 *>(s_beta + s0 + 4);
            const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
            float w8[8], d8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int s3 = s0 + u;
                const float bs = bv[u];
                w8[u] = (s3 < r) ? tv[u] * bs : 0.f;
                d8[u] = (s3 == r) ? bs : w8[u];
            }
            if ((r >> 3) >= 2 * (s0 >> 4))     // a row group that the packing holds
                __stcs(reinterpret_cast<uint4 *>(rec + R_T + tri_off(r, s0)), pack_bf8(w8));
            // rows 64..127 of the M = 128 operand repeat rows 0..63, so that every
            // TMEM lane quarter of the W accumulator holds real rows
            const uint4 pd = pack_h8(d8);
            *reinterpret_cast<uint4 *>(sm + SA_T + km_bf16(r, s0, 1024)) = pd;
            *reinterpret_cast<uint4 *>(sm + SA_T + km_bf16(64 + r, s0, 1024)) = pd;
        }
        fence_proxy_async_smem();
        sync_tc();

        // ===== W = T Diag(beta) K0: D_W[r][i] (M = 128, rows 64..127 a copy),
        // A = T Diag(beta) (K-major), B = K0 (MN-major)
        if (t == 0) {
            const uint32_t idw = instr_desc(kFmtF16, 128, 128, 0, 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t a = smem_desc(smem_u32(sm + SA_T + 256 * kk), 128, 1024, kSwizzleNone);
                const uint64_t b = smem_desc(smem_u32(sm + SA_K0 + 2048 * kk), 8192, 1024, kSwizzle128B);
                mma_bf16_ss(tmem + TMA_W, a, b, idw, kk > 0);
            }
            mma_commit(bar_mma);
        }
        if (!wait_all(bar_mma, 1)) { failed = true; fail_at = 3; fail_it = it; fail_next = has_next; break; }
    }
    {
        tc_fence_after();
        // the Khat / solve space is free: the next job's g
        if (t == 0 && has_next) issue_g(Jn);
        // ===== -W (bf16, K-major sw) -> the free K0 tile -> record rows 0..63
        // of both halves by two bulk copies.  TMEM lane l holds row l & 63 (the
        // two lane halves are copies); thread: row r, 32 channels
        {
            const int r = (32 * (warp & 3) + lane) & 63;
            const int cq = 2 * (warp >> 2) + ((warp & 3) >> 1);   // 32-channel quarter
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                float d[16];
                tmem_ld16(tmem + lane_base + TMA_W + 32 * cq + 16 * q2, d);
                tmem_wait_ld();
#pragma unroll
                for (int c8 = 0; c8 < 2; ++c8) {
                    float x8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x8[e] = -d[8 * c8 + e];
                    *reinterpret_cast<uint4 *>(sm + SA_K0 + sw_chunk(r, 4 * cq + 2 * q2 + c8, 8192)) =
                        pack_h8(x8);
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (t == 0) {
            bulk_store(rec + R_WQ, sm + SA_K0, 8192);
            bulk_store(rec + R_WQ + 16384, sm + SA_K0 + 8192, 8192);
            bulk_commit();
        }
    }
    // end of the job: every TMEM read and shared-memory use is done
    tc_fence_before();
    __syncthreads();
    if (!has_next) break;
    J = Jn;
    job = job_next;
    }   // job loop

    if (t == 0) bulk_wait();                 // record copies complete before the CTA exits
    if (t == 32) cp_async_wait_all();
    if (failed) {
        if (t == 0) atomicOr(&g_kda_device_error, 1u);
        // let copies and MMAs in flight finish (bounded) before freeing TMEM
        const uint32_t par = (uint32_t)(fail_it & 1);
        if (fail_at == 1) {
            mbar_wait(bar_qk, par, kWaitLimit);
            mbar_wait(bar_g, par, kWaitLimit);
        } else {
            mbar_wait(bar_mma, fail_at == 2 ? 0u : 1u, kWaitLimit);
            if (fail_at == 3 && fail_next) mbar_wait(bar_qk, par ^ 1u, kWaitLimit);
        }
    }
    sync_tc();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ============================================================================
// state pass: one CTA per (sequence, head), warp-specialised: 16 epilogue
// warps (512 threads, four per TMEM lane quarter), one warp that issues the
// MMAs and one that issues the copies, so that neither issue stream waits
// behind the other or behind the epilogues.
// ============================================================================
constexpr int NEPI = 512;                 // epilogue threads
constexpr int T_MMA = NEPI;               // the MMA-issuing thread (warp 16)
constexpr int T_TMA = NEPI + 32;          // the copy-issuing thread (warp 17)
constexpr int NTB = NEPI + 64;
constexpr uint32_t SB_WQ = 0;             // [-W ; Q0] (bulk copy 1, with T')
constexpr uint32_t SB_T = 32768;          // T' (packed triangle)
constexpr uint32_t SB_A = 37888;          // A' (packed triangle; bulk copy 2, with Kbar)
constexpr uint32_t SB_KB = 43008;         // Kbar (MN-major, 128B swizzle: 1 KB aligned)
constexpr uint32_t SB_VEC = 59392;        // 2 x 1 KB record vectors (double-buffered)
constexpr uint32_t SB_V = 92160;          // 16 KB: v chunk sw (TMA) = V^T, MN-major operand
                                          // 108544..141312 free: the fp16 copy of S^T lives in TMEM
constexpr uint32_t SB_O = 141312;         // 32 KB: o of even chunks, 4 x [64 r][32 j] fp32 (TMA store source)
constexpr uint32_t SB_GATE = 174080;      // 16 KB: gate chunk sw (TMA; gated variant only)
constexpr uint32_t SB_O1 = 190464;        // 32 KB: o of odd chunks
constexpr uint32_t SB_MISC = 223232;      // mbarriers at +0, +8, +16, +24, +40; TMEM base at +32; norm weight at +64
constexpr uint32_t SMEM_B_USED = SB_MISC + 576;
constexpr uint32_t SMEM_B_ALLOC = SMEM_B_USED + 1024;
static_assert(SB_T == R_T && SB_A == R_A && SB_KB == R_KB, "record pieces map onto shared memory");
static_assert(SB_KB == SB_A + kTriBytes && SB_KB % 1024 == 0, "A' then Kbar in one bulk copy; Kbar swizzle atoms aligned");
static_assert(SB_VEC + 2048 <= SB_V, "record vectors before v");
static_assert(SMEM_B_ALLOC <= 232448, "dynamic shared memory limit (227 KB)");
// TMEM columns: U^T | O^T | S^T master | S^T in fp16 | U^T in fp16.  Round 1
// writes [U | O] (N = 128) with the fp16 copy of S^T as its A operand;
// round 2 accumulates O (N = 64, B = A') and S (N = 128, B = Kbar) with the
// fp16 U^T as A.
constexpr uint32_t TMB_U = 0;             // U^T, 64 columns
constexpr uint32_t TMB_O = 64;            // O^T, 64 columns
constexpr uint32_t TMB_S = 128;           // S^T master fp32 (lane j, column i), 128 columns
constexpr uint32_t TMB_SB = 256;          // S^T in fp16 (lane j, column i / 2: pairs i, i + 1), 64 columns
constexpr uint32_t TMB_UP = 320;          // U^T as fp16 pairs (s, s + 1 per column): round 2's A, 32 columns
constexpr uint32_t TMEM_COLS_B = 512;
constexpr uint32_t COPY1 = R_A - R_WQ;    // bytes of [-W ; Q0] + T'
constexpr uint32_t COPY2 = R_VEC - R_A;   // bytes of A' + Kbar

// 16 consecutive floats of a record vector (16-byte aligned) in four
// broadcast 16-byte shared-memory loads
__device__ __forceinline__ void ld_vec16(const float *p, float (&x)[16]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float4 f = reinterpret_cast<const float4 *>(p)[c];
        x[4 * c] = f.x;
        x[4 * c + 1] = f.y;
        x[4 * c + 2] = f.z;
        x[4 * c + 3] = f.w;
    }
}

// barrier among the 512 epilogue threads only
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

// w / (1 + e^-x) for a channel pair: e^-x = 2^(-x log2 e) on the
// special-function unit (its scaling one packed multiply), the hardware
// reciprocal (a few ulp; e^-x overflowing to inf gives 0)
__device__ __forceinline__ float2 gate_sigmoid_w(float2 x, float2 w) {
    const float2 a = __fmul2_rn(x, make_float2(-1.4426950408889634f, -1.4426950408889634f));
    const float2 d = __fadd2_rn(make_float2(1.f, 1.f), make_float2(ex2_approx(a.x), ex2_approx(a.y)));
    return __fmul2_rn(w, make_float2(rcp_fast(d.x), rcp_fast(d.y)));
}

// GATED: the layer's output epilogue ("Colibri Kimi K3 Metal backend",
// section 8.4) on every row of o before it is stored: o / sqrt(mean_j o_j^2
// + eps) * norm_w_j * sigmoid(gate_j), the gate chunk arriving by TMA.
//
// Per chunk j (the block meets at two barriers, "mid" and "end"):
//   MMA warp:  wait record A(j) -> round 1 | mid | wait record B(j) -> round 2 | end
//   epilogue:  u = D_U + beta v in TMEM | mid | stage o(j-1) (gated:
//              normalise it) while round 2 runs; o(j) into registers, bf16
//              pieces of S and S <- Diag(e^{b_L(j+1)}) S for the next chunk | end
//   copy warp: request the gate of chunk j-1; after round 1, record A(j+1)
//              | mid | v(j+1); once staged, store o(j-1); after round 2,
//              record B(j+1) | end
template <bool GATED>
__global__ void __launch_bounds__(NTB, 1)
state_pass_kernel(const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                  const float *__restrict__ S0,
                  float *__restrict__ o, float *__restrict__ S_out, const int32_t *__restrict__ cu,
                  const int32_t *__restrict__ chunk_off, int N, int H, int max_chunks,
                  const uint8_t *__restrict__ recs, const __grid_constant__ CUtensorMap map_gate,
                  const float *__restrict__ norm_w, float norm_eps, int T) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar_a = reinterpret_cast<uint64_t *>(sm + SB_MISC);
    uint64_t *bar_b = bar_a + 1;
    uint64_t *bar_mma = bar_a + 2;            // round 1 completes phases of parity 0, round 2 parity 1
    uint64_t *bar_gate = bar_a + 3;           // gated variant: the gate chunk
    uint64_t *bar_ost = bar_a + 5;            // o of a chunk is staged (512 arrivals)
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + SB_MISC + 32);
    float *s_normw = reinterpret_cast<float *>(sm + SB_MISC + 64);
    __shared__ int s_seq;

    const int t = threadIdx.x;
    const int warp = t >> 5;
    const bool epi = t < NEPI;
    const int ch = t & 127;                   // epilogue: TMEM lane j = ch
    const int qt = (t >> 7) & 3;              // epilogue: column quarter
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;

    const int h = blockIdx.x % H;
    const int rank = blockIdx.x / H;
    const int n = lpt_sequence(cu, N, rank, &s_seq);
    const int tok0 = cu[n];
    const int len = cu[n + 1] - tok0;
    const size_t st_off = ((size_t)n * H + h) * kDK * kDV;
    const int cbase = chunk_off[n];
    int nch = len > 0 ? (len + C - 1) / C : 0;
    bool failed = false;
    if (chunk_off[n + 1] - cbase != nch || chunk_off[n + 1] > max_chunks) {
        nch = 0;                          // the plan does not match the workspace
        failed = true;
    }

    if (warp == 0) tmem_alloc(s_tmem, TMEM_COLS_B);
    if (t == 0) {
        mbar_init(bar_a, 1);
        mbar_init(bar_b, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_gate, 1);
        mbar_init(bar_ost, NEPI);
        fence_mbar_init();
        prefetch_tmap(&map_v);
        prefetch_tmap(&map_o);
        if (GATED) prefetch_tmap(&map_gate);
    }
    if (GATED && t < kDV) s_normw[t] = norm_w[t];
    sync_tc();
    const uint32_t tmem = *s_tmem;

    // ---- initial state: S^T master in TMEM (lane j, column i) + its fp16 copy
    if (epi) {
        float sv[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int i = 32 * qt + c;
            sv[c] = S0 ? S0[st_off + (size_t)i * kDV + ch] : 0.f;
        }
        float a[16], b2[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            a[c] = sv[c];
            b2[c] = sv[16 + c];
        }
        tmem_st16(tmem + lane_base + TMB_S + 32 * qt, a);
        tmem_st16(tmem + lane_base + TMB_S + 32 * qt + 16, b2);
        float pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = __uint_as_float(pack_h2(sv[2 * c], sv[2 * c + 1]));
        tmem_st16(tmem + lane_base + TMB_SB + 16 * qt, pk);
        tmem_wait_st();
    }
    fence_proxy_async_smem();
    sync_tc();

    // requests made by the copy thread, counted where they are made, so that
    // if a bounded wait gives up it waits for exactly what is in flight
    int issued_a = 0, issued_b = 0, issued_gate = 0, issued_mma = 0;
    auto rec_at = [&](int j) -> const uint8_t * {
        const int gc = KDA_DBG_INDEX(g_kda_device_error, cbase + j, 0, max_chunks);
        return recs + ((size_t)gc * H + h) * REC_BYTES;
    };
    // record A of chunk j and e^{b_L} of chunk j + 1 (for the scaling of S at
    // the end of chunk j), with the byte count of v, which issue_v requests
    // once the previous chunk's v is consumed
    auto issue_a = [&](int j) {
        const uint8_t *r = rec_at(j);
        mbar_arrive_expect_tx(bar_a, COPY1 + 1024 + 16384);
        ++issued_a;
        bulk_load(sm + SB_WQ, r + R_WQ, COPY1, bar_a);
        bulk_load(sm + SB_VEC + 1024 * (j & 1), r + R_VEC, 1024, bar_a);
    };
    auto issue_v = [&](int j) {
        tma_load_3d(sm + SB_V, &map_v, bar_a, 0, h, tok0 + j * C);
        tma_load_3d(sm + SB_V + 8192, &map_v, bar_a, 64, h, tok0 + j * C);
    };
    auto issue_gate = [&](int j) {
        mbar_arrive_expect_tx(bar_gate, 16384);
        ++issued_gate;
        tma_load_3d(sm + SB_GATE, &map_gate, bar_gate, 0, h, tok0 + j * C);
        tma_load_3d(sm + SB_GATE + 8192, &map_gate, bar_gate, 64, h, tok0 + j * C);
    };
    auto issue_b = [&](int j) {
        mbar_arrive_expect_tx(bar_b, COPY2);
        ++issued_b;
        bulk_load(sm + SB_A, rec_at(j) + R_A, COPY2, bar_b);
    };
    auto prefetch2 = [&](int j) {            // chunk j toward L2
        bulk_prefetch_l2(rec_at(j), REC_BYTES);
        tma_prefetch_l2_3d(&map_v, 0, h, tok0 + j * C);
        tma_prefetch_l2_3d(&map_v, 64, h, tok0 + j * C);
    };
    if (t == T_TMA && nch > 0) {
        issue_a(0);
        issue_v(0);
        issue_b(0);
        if (GATED) issue_gate(0);
        if (nch > 1) prefetch2(1);
    }
    bool bad = false;
    float po[16];                             // epilogue: o of the previous chunk

    // stage o of chunk jp from po (gated: normalise the rows); epilogue threads
    auto stage_o = [&](int jp) {
        const int Lp = min(C, len - jp * C);
        const uint32_t sbp = (jp & 1) ? SB_O1 : SB_O;
        const size_t row0 = (size_t)(tok0 + jp * C);
        if (GATED || Lp == C) {
            float *so = reinterpret_cast<float *>(sm + sbp + 8192 * (ch >> 5)) + (ch & 31);
#pragma unroll
            for (int k = 0; k < 16; ++k) so[(16 * qt + k) * 32] = po[k];
        } else {
            // the last, partial chunk of a sequence goes out row by row so
            // that the next sequence's rows are never written
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int r = 16 * qt + k;
                if (r < Lp) o[((size_t)KDA_DBG_INDEX(g_kda_device_error, (long long)(row0 + r), 0, T) * H + h) * kDV + ch] = po[k];
            }
        }
        if (GATED) {
            // per row: RMSNorm over the 128 columns times the weighted gate.
            // Thread: row rr, columns 32 m + 4 p8 .. +3 of the four boxes m.
            const int rr = t >> 3, p8 = t & 7;
            float4 gw[4];
            if (!mbar_wait(bar_gate, (uint32_t)(jp & 1), kWaitLimit)) bad = true;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int cg = (m & 1) * 4 + (p8 >> 1);          // 16-byte chunk of the gate row
                const uint2 gu = *reinterpret_cast<const uint2 *>(
                    sm + SB_GATE + 8192 * (m >> 1) + rr * 128 + ((cg ^ (rr & 7)) << 4) + 8 * (p8 & 1));
                const float2 ga = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&gu.x));
                const float2 gb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&gu.y));
                const float4 wv = *reinterpret_cast<const float4 *>(s_normw + 32 * m + 4 * p8);
                const float2 sa = gate_sigmoid_w(ga, make_float2(wv.x, wv.y));
                const float2 sb = gate_sigmoid_w(gb, make_float2(wv.z, wv.w));
                gw[m] = make_float4(sa.x, sa.y, sb.x, sb.y);
            }
            epi_sync();                          // every row of o is staged
            float4 x[4];
            float ss = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                x[m] = *reinterpret_cast<const float4 *>(sm + sbp + 8192 * m + rr * 128 + 16 * p8);
                ss = fmaf(x[m].x, x[m].x, fmaf(x[m].y, x[m].y, fmaf(x[m].z, x[m].z, fmaf(x[m].w, x[m].w, ss))));
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            ss += __shfl_xor_sync(0xffffffffu, ss, 4);
            const float rs = rsqrtf(ss * (1.f / 128.f) + norm_eps);
            const float2 rs2 = make_float2(rs, rs);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float2 ya = __fmul2_rn(__fmul2_rn(make_float2(x[m].x, x[m].y), rs2), make_float2(gw[m].x, gw[m].y));
                const float2 yb = __fmul2_rn(__fmul2_rn(make_float2(x[m].z, x[m].w), rs2), make_float2(gw[m].z, gw[m].w));
                const float4 y = make_float4(ya.x, ya.y, yb.x, yb.y);
                if (Lp == C)
                    *reinterpret_cast<float4 *>(sm + sbp + 8192 * m + rr * 128 + 16 * p8) = y;
                else if (rr < Lp)
                    *reinterpret_cast<float4 *>(
                        o + ((size_t)KDA_DBG_INDEX(g_kda_device_error, (long long)(row0 + rr), 0, T) * H + h) * kDV +
                        32 * m + 4 * p8) = y;
            }
        }
        fence_proxy_async_smem();
    };
    auto store_o = [&](int jp) {             // copy thread, after the barrier that follows stage_o
        if (min(C, len - jp * C) == C) {
            const uint32_t sbp = (jp & 1) ? SB_O1 : SB_O;
#pragma unroll
            for (int bx = 0; bx < 4; ++bx) tma_store_3d(&map_o, sm + sbp + 8192 * bx, 32 * bx, h, tok0 + jp * C);
            bulk_commit();
        }
    };

    for (int j = 0; j < nch; ++j) {
        const uint32_t par = (uint32_t)(j & 1);
        const float *vec = reinterpret_cast<const float *>(sm + SB_VEC + 1024 * par);

        // ===== round 1: D_U = -(W S)^T + (T' V)^T, D_O = (Q0 S)^T ============
        if (t == T_MMA) {
            if (mbar_wait(bar_a, par, kWaitLimit)) {
                tc_fence_after();
                const uint32_t id1 = instr_desc(kFmtF16, 128, 128, 0, 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t bw = smem_desc(
                        smem_u32(sm + SB_WQ + (uint32_t)(kk >> 2) * 16384 + (uint32_t)(kk & 3) * 32), 16,
                        1024, kSwizzle128B);
                    mma_bf16_ts(tmem + TMB_U, tmem + TMB_SB + 8 * kk, bw, id1, kk > 0);
                }
                // (T' V)^T: K-step kk meets only rows r >= 16 kk of the packed T'
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t idv = instr_desc(kFmtBF16, 128, 64 - 16 * kk, 1, 0);
                    const uint64_t av = smem_desc(smem_u32(sm + SB_V + 2048 * kk), 8192, 1024, kSwizzle128B);
                    const uint64_t bt = smem_desc(smem_u32(sm + SB_T + tri_base(kk)), 128, 256, kSwizzleNone);
                    mma_bf16_ss(tmem + TMB_U + 16 * kk, av, bt, idv, 1);
                }
                mma_commit(bar_mma);
                ++issued_mma;
            } else {
                bad = true;
            }
        }
        if (t == T_TMA) {
            // the buffer o(j - 1) is staged into was last read by the store of chunk j - 3
            bulk_wait_read_but_last();
            if (GATED && j >= 2) issue_gate(j - 1);
            // once round 1 has read them: the next chunk's round-1 operands
            if (!mbar_wait(bar_mma, 0u, kWaitLimit)) bad = true;   // round 1 may still read them
            else if (j + 1 < nch) issue_a(j + 1);
        }
        float uv[16];
        if (epi) {
            if (!mbar_wait(bar_a, par, kWaitLimit)) bad = true;   // vec and v of this chunk
            __syncwarp();
            {
                // S <- Diag(e^{b_L}) S for this chunk's round 2, while round 1
                // runs (it reads only the fp16 copy): off the serial chain
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t col = 32 * qt + 16 * hh;
                    float sv[16], eb[16];
                    tmem_ld16(tmem + lane_base + TMB_S + col, sv);
                    ld_vec16(vec + 128 + col, eb);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; ++c) sv[c] *= eb[c];
                    tmem_st16(tmem + lane_base + TMB_S + col, sv);
                }
            }
            // ===== u = D_U + beta v; round 2's A operand U^T as fp16 pairs =====
            float bt[16], vv[16];
            ld_vec16(vec + 16 * qt, bt);
#pragma unroll
            for (int k = 0; k < 16; ++k) vv[k] = bf(sm + SB_V + sw_elem64(16 * qt + k, ch));
            if (!mbar_wait(bar_mma, 0u, kWaitLimit)) bad = true;
            __syncwarp();
            tc_fence_after();
            tmem_ld16(tmem + lane_base + TMB_U + 16 * qt, uv);
            tmem_wait_ld();
            float up[8];
            bool u_big = false;               // |u| beyond fp16's finite range (or NaN)
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                uv[k] = fmaf(bt[k], vv[k], uv[k]);
                u_big |= !(fabsf(uv[k]) < 65504.f);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) up[c] = __uint_as_float(pack_h2(uv[2 * c], uv[2 * c + 1]));
            tmem_st8(tmem + lane_base + TMB_UP + 8 * qt, up);
            if (__any_sync(0xffffffffu, u_big) && (t & 31) == 0) atomicOr(&g_kda_device_error, kErrFp16Range);
            tmem_wait_st();
        }
        tc_fence_before();
        if (__syncthreads_or(bad)) {                            // ---- mid
            failed = true;
            break;
        }
        tc_fence_after();

        // ===== round 2: D_O += U^T A'^T (N = 64, A' K-major), S^T += U^T Kbar
        // (N = 128, Kbar MN-major); fp16, U^T from TMEM
        if (t == T_MMA) {
            if (mbar_wait(bar_b, par, kWaitLimit)) {
                const uint32_t idk = instr_desc(kFmtF16, 128, 128, 0, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    // K-step kk meets only rows r >= 16 kk of the packed A'
                    const uint32_t ida = instr_desc(kFmtF16, 128, 64 - 16 * kk, 0, 0);
                    const uint64_t ba = smem_desc(smem_u32(sm + SB_A + tri_base(kk)), 128, 256, kSwizzleNone);
                    const uint64_t bk = smem_desc(smem_u32(sm + SB_KB + 2048 * kk), 8192, 1024, kSwizzle128B);
                    mma_bf16_ts(tmem + TMB_O + 16 * kk, tmem + TMB_UP + 8 * kk, ba, ida, 1);
                    mma_bf16_ts(tmem + TMB_S, tmem + TMB_UP + 8 * kk, bk, idk, 1);
                }
                mma_commit(bar_mma);
                ++issued_mma;
            } else {
                bad = true;
            }
        }
        if (t == T_TMA) {
            // v is consumed: the next chunk's, and the chunk after it toward
            // L2 (the records are single-buffered in shared memory)
            if (j + 1 < nch) issue_v(j + 1);
            if (j + 2 < nch) prefetch2(j + 2);
            if (j > 0) {                     // o of the previous chunk, once staged
                if (mbar_wait(bar_ost, (uint32_t)((j - 1) & 1), kWaitLimit)) store_o(j - 1);
                else bad = true;
            }
            if (!mbar_wait(bar_mma, 1u, kWaitLimit)) bad = true;   // round 2 may still read them
            else if (j + 1 < nch) issue_b(j + 1);                    // A' and Kbar are consumed
        }

        // ===== the previous chunk's o is staged while round 2 runs; then
        // o = D_O + (q.k) u into registers, the fp16 copy of the new S^T, and
        // S <- Diag(e^{b_L}) S for the next chunk
        if (epi) {
            if (j > 0) {
                stage_o(j - 1);
                mbar_arrive(bar_ost);        // the copy thread stores it now
            }
            float qk[16];
            ld_vec16(vec + 64 + 16 * qt, qk);
            const bool next = j + 1 < nch;
            if (!mbar_wait(bar_mma, 1u, kWaitLimit)) bad = true;
            __syncwarp();
            tc_fence_after();
            {
                float ov[16];
                tmem_ld16(tmem + lane_base + TMB_O + 16 * qt, ov);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) po[k] = fmaf(qk[k], uv[k], ov[k]);
            }
            {
                if (next) {
                    float sv[32], pk[16];
                    tmem_ld32(tmem + lane_base + TMB_S + 32 * qt, sv);
#pragma unroll
                    for (int c = 0; c < 16; ++c) pk[c] = __uint_as_float(pack_h2(sv[2 * c], sv[2 * c + 1]));
                    tmem_st16(tmem + lane_base + TMB_SB + 16 * qt, pk);
                }
            }
            tmem_wait_st();
        }
        tc_fence_before();
        if (__syncthreads_or(bad)) { failed = true; break; }   // ---- end
    }
    // the last two chunks' o
    if (!failed && nch > 0) {
        if (t == T_TMA) {
            bulk_wait_read_but_last();
            if (GATED && nch >= 2) issue_gate(nch - 1);
        }
        __syncthreads();
        if (epi) stage_o(nch - 1);
        if (__syncthreads_or(bad)) failed = true;
        else if (t == T_TMA) store_o(nch - 1);
    }
    if (t == T_TMA) bulk_wait();             // o stores complete before the CTA exits

    if (failed) {
        if (t == T_TMA || t == 0) atomicOr(&g_kda_device_error, 1u);
        // let copies and MMAs in flight finish (bounded) before freeing TMEM
        if (t == T_TMA) {
            if (issued_a) mbar_wait(bar_a, (uint32_t)(issued_a - 1) & 1u, kWaitLimit);
            if (issued_b) mbar_wait(bar_b, (uint32_t)(issued_b - 1) & 1u, kWaitLimit);
            if (issued_gate) mbar_wait(bar_gate, (uint32_t)(issued_gate - 1) & 1u, kWaitLimit);
        }
        if (t == T_MMA && issued_mma) mbar_wait(bar_mma, (uint32_t)(issued_mma - 1) & 1u, kWaitLimit);
    } else if (epi) {
        // ---- final state: S_out[i][j] from the TMEM master (lane j, column i)
        tc_fence_after();
        float sv[32];
        tmem_ld32(tmem + lane_base + TMB_S + 32 * qt, sv);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int i = 32 * qt + c;
            S_out[st_off + (size_t)i * kDV + ch] = sv[c];
        }
    }
    sync_tc();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS_B);
}

// ---- per-device state the library keeps between calls --------------------
// Everything cached here belongs to one CUDA context of the device: a
// cudaDeviceReset destroys it (the pool, the kernel attributes, the scratch
// array's address), so each entry remembers the context it was made in and
// is made again when the current context differs.
constexpr int kMaxDevices = 64;

// Unique (for the process's lifetime) identity of the calling thread's
// current context; 0 when none is current or the driver cannot say.
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_cur || !get_id) return 0;
    CUcontext c = nullptr;
    if (get_cur(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

int current_device_checked(cudaError_t *e) {
    int dev = 0;
    *e = cudaGetDevice(&dev);
    if (*e == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) *e = cudaErrorInvalidDevice;
    return dev;
}

// The workspace pool: a library-owned stream-ordered pool per device that
// keeps its memory between calls (release threshold = max), so only the
// first call of a given size reaches the driver's allocator.
std::mutex g_pool_mu;
struct {
    unsigned long long ctx;
    cudaMemPool_t pool;
} g_pool[kMaxDevices] = {};

cudaError_t ws_alloc(void **p, size_t bytes, cudaStream_t s) {
    cudaError_t e;
    const int dev = current_device_checked(&e);
    if (e != cudaSuccess) return e;
    cudaMemPool_t pool;
    {
        std::lock_guard<std::mutex> lk(g_pool_mu);
        const unsigned long long ctx = current_context_id();
        if (!g_pool[dev].pool || (ctx != 0 && ctx != g_pool[dev].ctx)) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            cudaMemPool_t np = nullptr;
            e = cudaMemPoolCreate(&np, &props);
            if (e != cudaSuccess) return e;
            uint64_t thr = ~0ull;
            cudaMemPoolSetAttribute(np, cudaMemPoolAttrReleaseThreshold, &thr);
            g_pool[dev].pool = np;
            g_pool[dev].ctx = current_context_id();
        }
        pool = g_pool[dev].pool;
    }
    return cudaMallocFromPoolAsync(p, bytes, pool, s);
}

// The kernels' dynamic shared-memory limits, set once per device context.
std::mutex g_attr_mu;
unsigned long long g_attr_ctx[kMaxDevices] = {};

}  // namespace

// Workspace: chunk_off [N + 1] int32 and the job counter, the chunk table
// [max_chunks] int2 (each padded to 1 KB), then the records.
static size_t plan_bytes(int N, int64_t max_chunks) {
    return (((size_t)(N + 2) * sizeof(int32_t) + 1023) & ~(size_t)1023) +
           (((size_t)max_chunks * sizeof(int2) + 1023) & ~(size_t)1023);
}

size_t prefill_split_workspace_bytes(int N, int64_t T, int H) {
    const int64_t max_chunks = (T + C - 1) / C + N;
    return plan_bytes(N, max_chunks) + (size_t)max_chunks * (size_t)H * REC_BYTES;
}

namespace {

// Persistent intra-chunk grid: two CTAs per SM, at most one per job.
unsigned intra_grid(int64_t jobs) {
    static int sms[kMaxDevices] = {};
    int dev = 0;
    int n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (sms[dev] > 0) n = sms[dev];
    }
    return (unsigned)std::min<int64_t>(jobs, 2 * (int64_t)n);
}

// The three launches of one prefill, with the workspace at `ws` (at least
// prefill_split_workspace_bytes(N, T, H) bytes).  With a gate, the state pass
// writes the gated RMSNorm of o to `o` instead of o itself.
cudaError_t run_split(const void *q, const void *k, const void *v, const float *g,
                      const float *beta, const float *S0, float *o, float *S_out,
                      const int32_t *cu_seqlens, int N, int64_t T, int H, void *ws,
                      cudaStream_t stream, cudaEvent_t const *ev = nullptr,
                      const void *gate = nullptr, const float *norm_w = nullptr,
                      float norm_eps = 0.f) {
    const int64_t max_chunks = (T + C - 1) / C + N;
    static MapCache maps;
    CUtensorMap mq, mk, mv, mg, mo, mgate;
    if (!maps.get(&mq, kMapBf16Sw, q, T, H) || !maps.get(&mk, kMapBf16Sw, k, T, H) ||
        !maps.get(&mv, kMapBf16Sw, v, T, H) || !maps.get(&mg, kMapF32Sw, g, T, H) ||
        !maps.get(&mo, kMapF32Plain, o, T, H))
        return cudaErrorInvalidValue;
    if (gate && !maps.get(&mgate, kMapBf16Sw, gate, T, H)) return cudaErrorInvalidValue;
    if (!gate) mgate = mv;                   // unused by the ungated kernel
    cudaError_t e;
    const int dev = current_device_checked(&e);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(g_attr_mu);
        const unsigned long long ctx = current_context_id();
        if (ctx == 0 || ctx != g_attr_ctx[dev]) {
            e = cudaFuncSetAttribute(intra_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)SMEM_A_ALLOC);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(state_pass_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_B_ALLOC);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(state_pass_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_B_ALLOC);
            if (e != cudaSuccess) return e;
            g_attr_ctx[dev] = current_context_id();
        }
    }
    int32_t *chunk_off = static_cast<int32_t *>(ws);
    int2 *tab = reinterpret_cast<int2 *>(static_cast<uint8_t *>(ws) +
                                         (((size_t)(N + 2) * sizeof(int32_t) + 1023) & ~(size_t)1023));
    uint8_t *recs = static_cast<uint8_t *>(ws) + plan_bytes(N, max_chunks);
    if (ev) cudaEventRecord(ev[0], stream);
    chunk_plan_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, N, (int)T, chunk_off, tab);
    if (ev) cudaEventRecord(ev[1], stream);
    intra_chunk_kernel<<<intra_grid(max_chunks * H), NTA, SMEM_A_ALLOC, stream>>>(
        mq, mk, mg, beta, tab, chunk_off, N, H, recs, (int)T, (int)max_chunks);
    if (ev) cudaEventRecord(ev[2], stream);
    if (gate)
        state_pass_kernel<true><<<(unsigned)((int64_t)N * H), NTB, SMEM_B_ALLOC, stream>>>(
            mv, mo, S0, o, S_out, cu_seqlens, chunk_off, N, H, (int)max_chunks, recs, mgate, norm_w,
            norm_eps, (int)T);
    else
        state_pass_kernel<false><<<(unsigned)((int64_t)N * H), NTB, SMEM_B_ALLOC, stream>>>(
            mv, mo, S0, o, S_out, cu_seqlens, chunk_off, N, H, (int)max_chunks, recs, mgate, nullptr,
            0.f, (int)T);
    if (ev) cudaEventRecord(ev[3], stream);
    return cudaGetLastError();
}

bool grid_fits(int N, int64_t T, int H) {
    const int64_t max_chunks = (T + C - 1) / C + N;
    return max_chunks * H < (int64_t(1) << 31) && max_chunks < (int64_t(1) << 31);
}

}  // namespace

cudaError_t launch_prefill_split(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const float *S0, float *o, float *S_out,
                                 const int32_t *cu_seqlens, int N, int64_t T, int H,
                                 cudaStream_t stream, cudaEvent_t const *events) {
    if (!grid_fits(N, T, H)) return cudaErrorInvalidValue;
    void *ws = nullptr;
    cudaError_t e = ws_alloc(&ws, prefill_split_workspace_bytes(N, T, H), stream);
    if (e != cudaSuccess) return e;
    e = run_split(q, k, v, g, beta, S0, o, S_out, cu_seqlens, N, T, H, ws, stream, events);
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    return e != cudaSuccess ? e : ef;
}

cudaError_t launch_prefill_split_gated(const void *q, const void *k, const void *v,
                                       const float *g, const float *beta, const float *S0,
                                       const void *gate, const float *norm_w, float eps,
                                       float *out, float *S_out, const int32_t *cu_seqlens, int N,
                                       int64_t T, int H, cudaStream_t stream,
                                       cudaEvent_t const *events) {
    if (!grid_fits(N, T, H)) return cudaErrorInvalidValue;
    void *ws = nullptr;
    cudaError_t e = ws_alloc(&ws, prefill_split_workspace_bytes(N, T, H), stream);
    if (e != cudaSuccess) return e;
    e = run_split(q, k, v, g, beta, S0, out, S_out, cu_seqlens, N, T, H, ws, stream, events, gate,
                  norm_w, eps);
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    return e != cudaSuccess ? e : ef;
}

// Trims the current device's workspace pool to nothing (memory that no
// allocation still holds goes back to the driver).
cudaError_t release_workspace_pool() {
    cudaError_t e;
    const int dev = current_device_checked(&e);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_pool_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_pool[dev].pool || (ctx != 0 && ctx != g_pool[dev].ctx)) return cudaSuccess;   // none in this context
    return cudaMemPoolTrimTo(g_pool[dev].pool, 0);
}

// The layer prefill: the conv prologue writes q, k, v (bf16) into the front
// of one pool allocation, the gated prefill's records follow them.
cudaError_t launch_prefill_layer(const void *xq, const void *xk, const void *xv, const float *conv_w,
                                 const void *conv_in, void *conv_out, const float *g,
                                 const float *beta, const float *S0, const void *gate,
                                 const float *norm_w, float q_scale, float l2_eps, float norm_eps,
                                 float *out, float *S_out, const int32_t *cu_seqlens, int N,
                                 int64_t T, int H, cudaStream_t stream) {
    if (!grid_fits(N, T, H)) return cudaErrorInvalidValue;
    const size_t qkv_bytes = ((size_t)T * H * kDK * 2 + 1023) & ~(size_t)1023;
    void *ws = nullptr;
    cudaError_t e = ws_alloc(&ws, 3 * qkv_bytes + prefill_split_workspace_bytes(N, T, H), stream);
    if (e != cudaSuccess) return e;
    uint8_t *q = static_cast<uint8_t *>(ws);
    e = launch_conv_prologue(xq, xk, xv, conv_w, conv_in, conv_out, q, q + qkv_bytes,
                             q + 2 * qkv_bytes, cu_seqlens, N, T, H, q_scale, l2_eps, stream);
    if (e == cudaSuccess)
        e = run_split(q, q + qkv_bytes, q + 2 * qkv_bytes, g, beta, S0, out, S_out, cu_seqlens, N,
                      T, H, q + 3 * qkv_bytes, stream, nullptr, gate, norm_w, norm_eps);
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    return e != cudaSuccess ? e : ef;
}

// ---- fixed scratch for kda_prefill_chunked_noalloc -------------------------
// A file-scope device array replaces the pool workspace for callers that may
// not allocate device memory during a call.  Nothing in it needs to start at
// zero: the plan kernel writes every chunk offset and the intra-chunk kernel
// every record before the state pass reads them.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mu;
struct {
    unsigned long long ctx;
    void *addr;
} g_scratch[kMaxDevices] = {};
}  // namespace

cudaError_t launch_prefill_split_ws(const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, const float *S0, float *o, float *S_out,
                                    const int32_t *cu_seqlens, int N, int64_t T, int H, void *ws,
                                    cudaStream_t stream) {
    if (!grid_fits(N, T, H) || !ws) return cudaErrorInvalidValue;
    return run_split(q, k, v, g, beta, S0, o, S_out, cu_seqlens, N, T, H, ws, stream);
}

cudaError_t launch_prefill_split_noalloc(const void *q, const void *k, const void *v,
                                         const float *g, const float *beta, const float *S0,
                                         float *o, float *S_out, const int32_t *cu_seqlens, int N,
                                         int64_t T, int H, cudaStream_t stream) {
    if (!grid_fits(N, T, H) || prefill_split_workspace_bytes(N, T, H) > kNoAllocScratchBytes)
        return cudaErrorInvalidValue;
    cudaError_t e;
    const int dev = current_device_checked(&e);
    if (e != cudaSuccess) return e;
    void *ws = nullptr;
    {
        // first call on a device (and again after a device reset made a new
        // context): look up the array's address, with the device current
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        const unsigned long long ctx = current_context_id();
        if (!g_scratch[dev].addr || ctx == 0 || ctx != g_scratch[dev].ctx) {
            void *addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
            if (e != cudaSuccess) return e;
            g_scratch[dev].addr = addr;
            g_scratch[dev].ctx = current_context_id();
        }
        ws = g_scratch[dev].addr;
    }
    return run_split(q, k, v, g, beta, S0, o, S_out, cu_seqlens, N, T, H, ws, stream);
}

cudaError_t read_device_error(unsigned int *code, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_kda_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || !reset) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_kda_device_error, &zero, sizeof(unsigned int));
}

}  // namespace kda
