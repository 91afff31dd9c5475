// Chunked KDA prefill on the 5th-generation tensor cores (tcgen05 + TMEM,
// operands staged by TMA), bf16 q/k/v, chunk 64, fp32 state.
//
// Math (the recurrence of "Colibri Kimi K3 Metal backend", architecture
// section, unrolled over a chunk of L <= 64 tokens; b_r = sum_{t<=r} g_t):
//   G^qk_rs = sum_c q_rc k_sc e^{b_rc - b_sc} (s <= r),  G^kk likewise (s < r)
//   T  = (I + Diag(beta) G^kk)^-1 (unit lower triangular),  T' = (T - I) Diag(beta)
//   W  = T' K0 + Diag(beta) K0,        K0_r = e^{b_r} k_r
//   U~ = T' V  + Diag(beta) V
//   U  = U~ - W S
//   O  = Q0 S + A' U + Diag(q_r.k_r) U, Q0_r = e^{b_r} q_r, A' = strictly lower G^qk
//   S <- Diag(e^{b_L}) S + Kbar^T U,    Kbar_s = e^{b_L - b_s} k_s
// The diagonal terms (beta_r v_r, beta_r K0_r, (q_r.k_r) u_r) are added in
// fp32 outside the MMAs so that the dominant per-token terms are never
// rounded to a 16-bit operand.
//
// Decay folding for the gated Gram matrices: with 16-row sub-blocks p and
// sigma_p = b at the last row of p, a row r in p and key s <= end(p) give
//   e^{b_r - b_s} = e^{b_r - sigma_p} * e^{sigma_p - b_s},
// where the first factor lies in [1, e^{75}] and the second in (0, 1] when
// g >= -5 (the model's gate bound); the query side uses one operand
// X = [q_r e^{b_r - sigma_p(r)} ; k_r e^{b_r - sigma_p(r)}] (128 rows) and
// the key side a stack of four operands Khat^(p)_s = k_s e^{sigma_p - b_s}
// (16(p+1) rows each, 160 in all): one M=128, N=160 MMA gives both Gram
// matrices, row r reading the column block of its own sub-block.
//
// Precision: MMAs that carry state-side terms (W S, Q0 S, the Gram and UT
// products) use kind::f16 with bf16 operands; MMAs that carry the fresh
// per-token terms (A' U and Kbar^T U) use kind::tf32 with operands rounded to
// nearest in software.  Accumulation is fp32 in TMEM; the state is kept in
// fp32 in TMEM for the whole sequence.
//
// One CTA (512 threads) per (sequence, head), walking its chunks in order;
// the MMAs are transposed so that M = 128 is always dk or dv:
//   D_G[128 x 160] = X . Khat^T             D_W[i][r]  = (T' K0)^T
//   D_U[j][r]      = (T' V)^T - (W S)^T     D_O[j][r]  = (Q0 S)^T + (A' U)^T
//   D_S[j][i]     += (Kbar^T U)^T            (S^T kept in TMEM, lane j, column i)
#include <cudaTypedefs.h>

#include "kda_internal.h"
#include "tc_layout.cuh"

namespace kda {

// Nonzero when a bounded wait inside the tensor-core kernel gave up.
__device__ unsigned int g_kda_device_error = 0;

namespace {
using namespace tc;

constexpr int C = 64;
constexpr int NT = 512;

// shared memory map (bytes from a 1024-aligned base).  "sw" = 128-byte
// swizzled canonical layout, "il" = interleaved (no swizzle) canonical layout.
constexpr uint32_t SM_STG_Q = 0;          // q chunk: 2 x [64 r][64 c] sw (TMA)
constexpr uint32_t SM_STG_K = 16384;      // k chunk: same
constexpr uint32_t SM_STG_V = 32768;      // v chunk: same = V^T, MN-major operand
constexpr uint32_t SM_X = 49152;          // 32 KB: Gram A [128][128] K-major sw | M fp32 [64][68] + solve temps | U^T tf32 K-major il
constexpr uint32_t SM_KH = 81920;         // 40 KB: Gram B Khat [160][128] K-major sw | A' (16K) + -W^T (16K) + T' (8K)
constexpr uint32_t SM_A = SM_KH;          //   A' tf32 K-major il [r][s], 16 KB
constexpr uint32_t SM_TB = SM_KH + 16384; //   -T Diag(beta) tf32 K-major il [r][s], 16 KB
constexpr uint32_t SM_T = SM_KH + 32768;  //   T' bf16 K-major il [r][s], 8 KB
constexpr uint32_t SM_Q0 = 122880;        // 16 KB: Q0 [64][128] K-major sw (with K0: next chunk's g, cp.async)
constexpr uint32_t SM_K0 = 139264;        // 16 KB: K0 [64 s][128 i] MN-major sw (A of the W product)
constexpr uint32_t SM_KB = 155648;        // 32 KB: Kbar^T [128 i][64 s] tf32 K-major il (B of the dS product)
constexpr uint32_t SM_S = 188416;         // 32 KB: S^T bf16 K-major il [j][i]
constexpr uint32_t SM_MISC = 221184;
constexpr uint32_t MISC_BETA = 0;         // float[64]
constexpr uint32_t MISC_GAM = 256;        // float[128]  e^{b_L}
constexpr uint32_t MISC_DQ = 768;         // float[64]   q_r . k_r (shared-memory atomics)
constexpr uint32_t MISC_TOT = 1024;       // float[4][128] sub-block totals, then carry - sigma_u
constexpr uint32_t MISC_SIG = 3072;       // float[4][128] local prefix at sub-block ends, then e^{b_L - sigma_u}
constexpr uint32_t MISC_DD = 5120;        // float[4][128] per-channel decay factors
constexpr uint32_t MISC_BETAN = 7168;     // float[64]   next chunk's beta (cp.async)
constexpr uint32_t MISC_EP = 7424;        // float[4][128] e^{sigma_u}
constexpr uint32_t MISC_BAR = 9472;       // 4 x u64 mbarriers
constexpr uint32_t MISC_TMEM = 9504;      // u32 TMEM base
constexpr uint32_t SMEM_USED = SM_MISC + 9520;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;   // alignment slack
static_assert(MISC_BAR + 32 <= MISC_TMEM, "mbarrier slots");
static_assert(SMEM_ALLOC <= 232448, "dynamic shared memory limit (227 KB)");
constexpr int MLD = 68;                   // row stride (floats) of M / T

// TMEM columns (512 allocated)
constexpr uint32_t TM_S = 0;      // S^T master fp32 (lane j, column i), 128 cols
constexpr uint32_t TM_DS = 128;   // (Kbar^T U)^T, 128 cols
constexpr uint32_t TM_G = 256;    // Gram D, 160 cols
constexpr uint32_t TM_P = 128;    // (K0 S)^T, 64 cols inside TM_DS (M1 -> M2)
constexpr uint32_t TM_U = 320;    // U D, 64 cols (after the Gram epilogue)
constexpr uint32_t TM_O = 448;    // O D, 64 cols

struct Bars {
    uint64_t *qk, *v, *mma, *g;
};

__device__ __forceinline__ void issue_load_qk(uint8_t *sm, const CUtensorMap *mq,
                                              const CUtensorMap *mk, uint64_t *bar, int h,
                                              int tok) {
    mbar_arrive_expect_tx(bar, 32768);
    tma_load_3d(sm + SM_STG_Q, mq, bar, 0, h, tok);
    tma_load_3d(sm + SM_STG_Q + 8192, mq, bar, 64, h, tok);
    tma_load_3d(sm + SM_STG_K, mk, bar, 0, h, tok);
    tma_load_3d(sm + SM_STG_K + 8192, mk, bar, 64, h, tok);
}
__device__ __forceinline__ void issue_load_v(uint8_t *sm, const CUtensorMap *mv, uint64_t *bar,
                                             int h, int tok) {
    mbar_arrive_expect_tx(bar, 16384);
    tma_load_3d(sm + SM_STG_V, mv, bar, 0, h, tok);
    tma_load_3d(sm + SM_STG_V + 8192, mv, bar, 64, h, tok);
}

__global__ void __launch_bounds__(NT, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_g,
                  const float *__restrict__ g,
                  const float *__restrict__ beta, const float *__restrict__ S0,
                  float *__restrict__ o, float *S_out, const int32_t *__restrict__ cu, int N,
                  int H) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *s_beta = reinterpret_cast<float *>(sm + SM_MISC + MISC_BETA);
    float *s_gam = reinterpret_cast<float *>(sm + SM_MISC + MISC_GAM);
    float *s_dq = reinterpret_cast<float *>(sm + SM_MISC + MISC_DQ);
    float *s_tot = reinterpret_cast<float *>(sm + SM_MISC + MISC_TOT);
    float *s_sig = reinterpret_cast<float *>(sm + SM_MISC + MISC_SIG);
    float *s_dd = reinterpret_cast<float *>(sm + SM_MISC + MISC_DD);
    float *s_ep = reinterpret_cast<float *>(sm + SM_MISC + MISC_EP);
    float *s_el = s_sig;             // reused once sigma is folded into the carries
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SM_MISC + MISC_BAR);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + SM_MISC + MISC_TMEM);
    __shared__ int s_seq;

    const int t = threadIdx.x;
    const int warp = t >> 5;
    const int lane = t & 31;
    const int ch = t & 127;          // TMEM lane (i or j) owned in the epilogues
    const int qt = t >> 7;           // column quarter owned in the epilogues
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    // operand-build layout: row rb of sub-blocks 2sp, 2sp+1; channels 8cc..8cc+7
    const int rb = lane & 15;
    const int cc = 2 * (warp & 7) + (lane >> 4);
    const int sp = warp >> 3;

    const int h = blockIdx.x % H;
    const int rank = blockIdx.x / H;
    const int n = lpt_sequence(cu, N, rank, &s_seq);
    const int tok0 = cu[n];
    const int len = cu[n + 1] - tok0;
    const size_t st_off = ((size_t)n * H + h) * kDK * kDV;

    Bars B{bars + 0, bars + 1, bars + 2, bars + 3};
    if (warp == 0) tmem_alloc(s_tmem, 512);
    if (t == 0) {
        mbar_init(B.qk, 1);
        mbar_init(B.v, 1);
        mbar_init(B.mma, 1);
        mbar_init(B.g, 1);
        fence_mbar_init();
        prefetch_tmap(&map_g);
        prefetch_tmap(&map_q);
        prefetch_tmap(&map_k);
        prefetch_tmap(&map_v);
    }
    sync_tc();
    const uint32_t tmem = *s_tmem;
    uint32_t mma_phase = 0;
    bool failed = false;

    // ---- initial state: S^T master in TMEM (lane j, column i) + bf16 copy
    {
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
        tmem_st16(tmem + lane_base + TM_S + 32 * qt, a);
        tmem_st16(tmem + lane_base + TM_S + 32 * qt + 16, b2);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
            float x8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x8[u] = sv[8 * c8 + u];
            *reinterpret_cast<uint4 *>(sm + SM_S + km_bf16(ch, 32 * qt + 8 * c8, 2048)) = pack_bf8(x8);
        }
        tmem_wait_st();
    }

    const int nchunks = (len + C - 1) / C;
    if (t == 0 && nchunks > 0) {
        issue_load_qk(sm, &map_q, &map_k, B.qk, h, tok0);
        issue_load_v(sm, &map_v, B.v, h, tok0);
    }
    // The next chunk's g ([64 rows][128 channels] fp32, four 128B-swizzled TMA
    // boxes of 32 channels) lands in the Q0/K0 region, which is free from the W
    // epilogue to the next operand build; beta (64 floats) is copied with
    // cp.async.  Rows past the end of the sequence are masked at use.
    float *s_betan = reinterpret_cast<float *>(sm + SM_MISC + MISC_BETAN);
    auto fetch_g = [&](int c0) {
        if (c0 >= len) return;
        if (t == 0) {
            mbar_arrive_expect_tx(B.g, 32768);
#pragma unroll
            for (int bx = 0; bx < 4; ++bx)
                tma_load_3d(sm + SM_Q0 + 8192 * bx, &map_g, B.g, 32 * bx, h, tok0 + c0);
        }
        if (t < C) {
            const float *src = beta + (size_t)(tok0 + min(c0 + t, len - 1)) * H + h;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(s_betan + t)), "l"(src) : "memory");
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
    };
    fetch_g(0);

    for (int ci = 0; ci < nchunks && !failed; ++ci) {
        const int c0 = ci * C;
        const int Lc = min(C, len - c0);
        const uint32_t par = (uint32_t)(ci & 1);

        // ===== B1: decay prefix sums and every intra-chunk operand ==========
        {
            asm volatile("cp.async.wait_all;" ::: "memory");
            if (!wait_all(B.g, par)) { failed = true; break; }
            const float betan = (t < C) ? s_betan[t] : 0.f;
            // column scan in place in the g tile: thread = (channel i, sub-block u);
            // element (r, c) of the tile: box c/32, 128-byte rows, swizzled chunks
            auto g_at = [&](int r, int c) -> float * {
                return reinterpret_cast<float *>(sm + SM_Q0 + 8192 * (c >> 5) + r * 128 +
                                                 ((((c & 31) >> 2) ^ (r & 7)) << 4) + (c & 3) * 4);
            };
            {
                const int i = t & 127, u = t >> 7;
                float acc = 0.f, at_last = 0.f;
                const int lastrow = min(16 * u + 15, Lc - 1);
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) {
                    const int r = 16 * u + rr;
                    float *pg = g_at(r, i);
                    acc += (r < Lc) ? *pg : 0.f;
                    *pg = acc;                             // local (sub-block) prefix
                    if (r == lastrow) at_last = acc;
                }
                s_tot[u * 128 + i] = acc;                  // sub-block total
                s_sig[u * 128 + i] = at_last;              // local prefix at its last valid row
            }
            if (t < C) {
                s_beta[t] = (t < Lc) ? betan : 0.f;
                s_dq[t] = 0.f;
            }
            __syncthreads();
            // per channel: carries, sigma_u = b at the last valid row of sub-block u,
            // d0 = e^{sigma_0}, dw = e^{sigma_w - sigma_{w-1}}, e^{sigma_u}, e^{b_L - sigma_u}
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
                    if (u == lu) bL = base[u] + s_sig[u * 128 + t];
#pragma unroll
                for (int u = 0; u < 4; ++u) sg[u] = (u <= lu) ? base[u] + s_sig[u * 128 + t] : bL;
#pragma unroll
                for (int u = 0; u < 4; ++u) s_tot[u * 128 + t] = base[u] - sg[u];   // carry - sigma_u
                const float d0 = __expf(sg[0]), d1 = __expf(sg[1] - sg[0]), d2 = __expf(sg[2] - sg[1]),
                            d3 = __expf(sg[3] - sg[2]);
                s_dd[t] = d0;
                s_dd[128 + t] = d1;
                s_dd[256 + t] = d2;
                s_dd[384 + t] = d3;
                const float e1 = d0 * d1, e2 = e1 * d2, e3 = e2 * d3;
                s_ep[t] = d0;
                s_ep[128 + t] = e1;
                s_ep[256 + t] = e2;
                s_ep[384 + t] = e3;
                const float l2 = d3, l1 = d2 * d3, l0 = d1 * l1;
                s_el[t] = l0;                              // s_sig of channel t is consumed
                s_el[128 + t] = l1;
                s_el[256 + t] = l2;
                s_el[384 + t] = 1.f;
                s_gam[t] = e3;
            }
            __syncthreads();
            // F = e^{b - sigma_u} in [1, e^75] for valid rows, b = local prefix + carry
            float b[2][8];
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const int u = 2 * sp + v;
                const int r = 16 * u + rb;
                const bool valid = r < Lc;
                const uint8_t *rowp = sm + SM_Q0 + 8192 * (cc >> 2) + r * 128;
                const int c4 = 2 * (cc & 3);
                const float4 ga = *reinterpret_cast<const float4 *>(rowp + ((c4 ^ (r & 7)) << 4));
                const float4 gb = *reinterpret_cast<const float4 *>(rowp + (((c4 + 1) ^ (r & 7)) << 4));
                const float4 ba = *reinterpret_cast<const float4 *>(s_tot + u * 128 + 8 * cc);
                const float4 bb = *reinterpret_cast<const float4 *>(s_tot + u * 128 + 8 * cc + 4);
                const float gl[8] = {ga.x + ba.x, ga.y + ba.y, ga.z + ba.z, ga.w + ba.w,
                                     gb.x + bb.x, gb.y + bb.y, gb.z + bb.z, gb.w + bb.w};
#pragma unroll
                for (int c = 0; c < 8; ++c) b[v][c] = valid ? __expf(gl[c]) : 0.f;
            }
            __syncthreads();          // the g tile is read: Q0/K0 may be written

            if (!wait_all(B.qk, par)) { failed = true; break; }
            float dd[4][8];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float4 da = *reinterpret_cast<const float4 *>(s_dd + w * 128 + 8 * cc);
                const float4 db = *reinterpret_cast<const float4 *>(s_dd + w * 128 + 8 * cc + 4);
                dd[w][0] = da.x; dd[w][1] = da.y; dd[w][2] = da.z; dd[w][3] = da.w;
                dd[w][4] = db.x; dd[w][5] = db.y; dd[w][6] = db.z; dd[w][7] = db.w;
            }
            float dqp[2];
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const int u = 2 * sp + v;
                const int r = 16 * u + rb;
                float qv[8], kv[8];
                unpack_bf8(*reinterpret_cast<const uint4 *>(sm + SM_STG_Q + sw_chunk(r, cc, 8192)), qv);
                unpack_bf8(*reinterpret_cast<const uint4 *>(sm + SM_STG_K + sw_chunk(r, cc, 8192)), kv);
                float G[8], xq[8], xk[8], ep[8], el[8];
                {
                    const float4 e0 = *reinterpret_cast<const float4 *>(s_ep + u * 128 + 8 * cc);
                    const float4 e1 = *reinterpret_cast<const float4 *>(s_ep + u * 128 + 8 * cc + 4);
                    const float4 l0 = *reinterpret_cast<const float4 *>(s_el + u * 128 + 8 * cc);
                    const float4 l1 = *reinterpret_cast<const float4 *>(s_el + u * 128 + 8 * cc + 4);
                    ep[0] = e0.x; ep[1] = e0.y; ep[2] = e0.z; ep[3] = e0.w;
                    ep[4] = e1.x; ep[5] = e1.y; ep[6] = e1.z; ep[7] = e1.w;
                    el[0] = l0.x; el[1] = l0.y; el[2] = l0.z; el[3] = l0.w;
                    el[4] = l1.x; el[5] = l1.y; el[6] = l1.z; el[7] = l1.w;
                }
                float dot = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    dot = fmaf(qv[c], kv[c], dot);
                    const float F = b[v][c];
                    G[c] = (F > 0.f) ? __fdividef(1.f, F) : 0.f;               // (0, 1]
                    xq[c] = qv[c] * F;
                    xk[c] = kv[c] * F;
                }
                dqp[v] = (r < Lc) ? dot : 0.f;
                // Gram A operand: q rows 0..63, k rows 64..127
                *reinterpret_cast<uint4 *>(sm + SM_X + sw_chunk(r, cc, 16384)) = pack_bf8(xq);
                *reinterpret_cast<uint4 *>(sm + SM_X + sw_chunk(64 + r, cc, 16384)) = pack_bf8(xk);
                // Khat stack: block pp >= u holds k_s e^{sigma_pp - b_s} at row 8pp(pp+1) + s
                float kh[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) kh[c] = kv[c] * G[c];
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    if (pp >= u) {
                        if (pp > u) {
#pragma unroll
                            for (int c = 0; c < 8; ++c) kh[c] *= dd[pp][c];
                        }
                        *reinterpret_cast<uint4 *>(sm + SM_KH + sw_chunk(8 * pp * (pp + 1) + r, cc, 20480)) =
                            pack_bf8(kh);
                    }
                }
                // Q0 = q e^{b}, K0 = k e^{b}, Kbar = k e^{b_L - b}
                float q0[8], k0[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    q0[c] = xq[c] * ep[c];
                    k0[c] = xk[c] * ep[c];
                }
                *reinterpret_cast<uint4 *>(sm + SM_Q0 + sw_chunk(r, cc, 8192)) = pack_bf8(q0);
                *reinterpret_cast<uint4 *>(sm + SM_K0 + sw_chunk(r, cc, 8192)) = pack_bf8(k0);
                // Kbar^T tf32 K-major il [i][s] (B of the dS product).  A 4x4
                // transpose inside each quad of lanes (4 consecutive rows) gives
                // every lane 4 consecutive s for channels 2b, 2b+1: 16-byte stores.
                {
                    float kbv[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) kbv[c] = kv[c] * G[c] * el[c];
                    const int bq = rb & 3;
                    float o0[4], o1[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // send the pair for destination lane (bq - k) & 3, receive from (bq + k) & 3
                        const int dst = (bq - k) & 3;
                        const float s0 = dst == 0 ? kbv[0] : dst == 1 ? kbv[2] : dst == 2 ? kbv[4] : kbv[6];
                        const float s1 = dst == 0 ? kbv[1] : dst == 1 ? kbv[3] : dst == 2 ? kbv[5] : kbv[7];
                        const int srcl = (lane & ~3) | ((bq + k) & 3);
                        const float r0 = __shfl_sync(0xffffffffu, s0, srcl);
                        const float r1 = __shfl_sync(0xffffffffu, s1, srcl);
                        const int srow = (bq + k) & 3;   // row offset of the received pair
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (e == srow) {
                                o0[e] = r0;
                                o1[e] = r1;
                            }
                        }
                    }
                    const int s0r = 16 * u + (rb & ~3);
                    const int i0 = 8 * cc + 2 * bq;
                    *reinterpret_cast<uint4 *>(sm + SM_KB + km_tf32(i0, s0r, 2048)) =
                        make_uint4(to_tf32(o0[0]), to_tf32(o0[1]), to_tf32(o0[2]), to_tf32(o0[3]));
                    *reinterpret_cast<uint4 *>(sm + SM_KB + km_tf32(i0 + 1, s0r, 2048)) =
                        make_uint4(to_tf32(o1[0]), to_tf32(o1[1]), to_tf32(o1[2]), to_tf32(o1[3]));
                }
            }
            // q_r . k_r: combine the two channel chunks of this warp, then
            // accumulate the eight warps of this row half in shared memory
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const float d2 = dqp[v] + __shfl_xor_sync(0xffffffffu, dqp[v], 16);
                if (lane < 16) atomicAdd(s_dq + 16 * (2 * sp + v) + rb, d2);
            }
        }
        fence_proxy_async_smem();
        sync_tc();

        // ===== M1: Gram (X Khat^T) and O1 = S^T Q0^T ========================
        // The three independent accumulators are issued interleaved so that
        // consecutive MMAs do not wait on one another.
        if (t == 0) {
            const uint32_t idg = instr_desc(kFmtBF16, 128, 160, 0, 0);
            const uint32_t ido = instr_desc(kFmtBF16, 128, 64, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ko = (uint32_t)(kk >> 2), kb2 = (uint32_t)(kk & 3) * 32u;
                const uint64_t ax = smem_desc(smem_u32(sm + SM_X + ko * 16384 + kb2), 16, 1024, kSwizzle128B);
                const uint64_t bk = smem_desc(smem_u32(sm + SM_KH + ko * 20480 + kb2), 16, 1024, kSwizzle128B);
                const uint64_t as = smem_desc(smem_u32(sm + SM_S + 256 * kk), 128, 2048, kSwizzleNone);
                const uint64_t bq = smem_desc(smem_u32(sm + SM_Q0 + ko * 8192 + kb2), 16, 1024, kSwizzle128B);
                const uint64_t bk0 = smem_desc(smem_u32(sm + SM_K0 + ko * 8192 + kb2), 16, 1024, kSwizzle128B);
                mma_bf16_ss(tmem + TM_G, ax, bk, idg, kk > 0);
                mma_bf16_ss(tmem + TM_O, as, bq, ido, kk > 0);
                // P^T = S^T K0^T (the W S product, with W = T Diag(beta) K0 applied in M2)
                mma_bf16_ss(tmem + TM_P, as, bk0, ido, kk > 0);
            }
            mma_commit(B.mma);
            // q/k staging is consumed: load the next chunk's q and k
            if (ci + 1 < nchunks) issue_load_qk(sm, &map_q, &map_k, B.qk, h, tok0 + c0 + C);
        }
        if (!wait_all(B.mma, mma_phase)) { failed = true; break; }
        mma_phase ^= 1;
        tc_fence_after();
        // Q0/K0 are consumed: fetch the next chunk's g and beta into that space
        fetch_g(c0 + C);

        // ===== E1: Gram epilogue -> A' (tf32) and M (fp32); diagonal dots ====
        // lane = row (0..63 q rows, 64..127 k rows); quarter qt = columns s in [16qt, 16qt+16)
        float *Mm = reinterpret_cast<float *>(sm + SM_X);
        {
            const bool qside = ch < 64;
            const int r = ch & 63;
            const int p = r >> 4;
            const int plo = (r >> 5) * 2;                      // sub-blocks of this warp's rows
            const uint32_t col_lo = (uint32_t)min(8 * plo * (plo + 1) + 16 * qt, 144);
            const uint32_t col_hi = (uint32_t)min(8 * (plo + 1) * (plo + 2) + 16 * qt, 144);
            float va[16], vb[16];
            tmem_ld16(tmem + lane_base + TM_G + col_lo, va);
            tmem_ld16(tmem + lane_base + TM_G + col_hi, vb);
            tmem_wait_ld();
            const bool use_hi = p != plo;
            const bool have = qt <= p && r < Lc;
            const float br = s_beta[r];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float x4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = 16 * qt + 4 * j + e;
                    const float val = use_hi ? vb[4 * j + e] : va[4 * j + e];
                    x4[e] = (have && s < r) ? val : 0.f;
                }
                if (qside) {
                    *reinterpret_cast<uint4 *>(sm + SM_A + km_tf32(r, 16 * qt + 4 * j, 2048)) =
                        make_uint4(to_tf32(x4[0]), to_tf32(x4[1]), to_tf32(x4[2]), to_tf32(x4[3]));
                } else {
                    *reinterpret_cast<float4 *>(Mm + r * MLD + 16 * qt + 4 * j) =
                        make_float4(br * x4[0], br * x4[1], br * x4[2], br * x4[3]);
                }
            }
        }
        __syncthreads();

        // ===== S1: T = (I + M)^-1 by 16-row blocks, in place; T' = (T-I)Diag(beta)
        {
            float *Yt = Mm + 64 * MLD;        // temporaries: 2 x [16][16], then [32][32]
            // diagonal blocks (I + M_pp)^-1 by forward substitution across a
            // 16-lane group: lane = row r, two right-hand sides (columns c0, c0+1)
            // per thread; step s broadcasts x_s and every row r > s applies M_rs
            {
                const int r = t & 15;
                const int grp = t >> 4;                 // 32 groups
                const int p = grp >> 3, c0 = 2 * (grp & 7);
                const float *Mr = Mm + (16 * p + r) * MLD + 16 * p;
                float mr[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(Mr + 4 * j);
                    mr[4 * j] = m4.x; mr[4 * j + 1] = m4.y; mr[4 * j + 2] = m4.z; mr[4 * j + 3] = m4.w;
                }
                float x0 = (r == c0) ? 1.f : 0.f, x1 = (r == c0 + 1) ? 1.f : 0.f;
#pragma unroll
                for (int s2 = 0; s2 < 15; ++s2) {
                    const float b0 = __shfl_sync(0xffffffffu, x0, s2, 16);
                    const float b1 = __shfl_sync(0xffffffffu, x1, s2, 16);
                    if (r > s2) {
                        x0 = fmaf(-mr[s2], b0, x0);
                        x1 = fmaf(-mr[s2], b1, x1);
                    }
                }
                __syncthreads();
                Mm[(16 * p + r) * MLD + 16 * p + c0] = x0;
                Mm[(16 * p + r) * MLD + 16 * p + c0 + 1] = x1;
            }
            __syncthreads();
            // off-diagonal blocks, two levels: (1) T_10 and T_32 (16x16 each,
            // T_pq = -T_pp M_pq T_qq); (2) the lower-left 32x32 block
            // T_C = -T_B M_C T_A with T_A, T_B the inverted 32x32 diagonal blocks
            if (t < 128) {
                const int blk = t >> 6, r = (t >> 2) & 15, c4 = t & 3;
                const int p = blk ? 3 : 1, q = p - 1;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                float arow[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(Mm + (16 * p + r) * MLD + 16 * q + 4 * j);
                    arow[4 * j] = a4.x; arow[4 * j + 1] = a4.y; arow[4 * j + 2] = a4.z; arow[4 * j + 3] = a4.w;
                }
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float a = arow[m];
                    const float4 tv = *reinterpret_cast<const float4 *>(Mm + (16 * q + m) * MLD + 16 * q + 4 * c4);
                    acc.x = fmaf(a, tv.x, acc.x);
                    acc.y = fmaf(a, tv.y, acc.y);
                    acc.z = fmaf(a, tv.z, acc.z);
                    acc.w = fmaf(a, tv.w, acc.w);
                }
                *reinterpret_cast<float4 *>(Yt + (blk * 16 + r) * 16 + 4 * c4) = acc;
            }
            __syncthreads();
            if (t < 128) {
                const int blk = t >> 6, r = (t >> 2) & 15, c4 = t & 3;
                const int p = blk ? 3 : 1, q = p - 1;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                float arow[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(Mm + (16 * p + r) * MLD + 16 * p + 4 * j);
                    arow[4 * j] = a4.x; arow[4 * j + 1] = a4.y; arow[4 * j + 2] = a4.z; arow[4 * j + 3] = a4.w;
                }
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float a = arow[m];
                    const float4 yv = *reinterpret_cast<const float4 *>(Yt + (blk * 16 + m) * 16 + 4 * c4);
                    acc.x = fmaf(a, yv.x, acc.x);
                    acc.y = fmaf(a, yv.y, acc.y);
                    acc.z = fmaf(a, yv.z, acc.z);
                    acc.w = fmaf(a, yv.w, acc.w);
                }
                *reinterpret_cast<float4 *>(Mm + (16 * p + r) * MLD + 16 * q + 4 * c4) =
                    make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
            }
            __syncthreads();
            if (t < 256) {
                // Y2 = M[32:64][0:32] T[0:32][0:32]
                const int r = t >> 3, c4 = t & 7;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                float arow[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(Mm + (32 + r) * MLD + 4 * j);
                    arow[4 * j] = a4.x; arow[4 * j + 1] = a4.y; arow[4 * j + 2] = a4.z; arow[4 * j + 3] = a4.w;
                }
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const float a = arow[m];
                    const float4 tv = *reinterpret_cast<const float4 *>(Mm + m * MLD + 4 * c4);
                    acc.x = fmaf(a, tv.x, acc.x);
                    acc.y = fmaf(a, tv.y, acc.y);
                    acc.z = fmaf(a, tv.z, acc.z);
                    acc.w = fmaf(a, tv.w, acc.w);
                }
                *reinterpret_cast<float4 *>(Yt + r * 32 + 4 * c4) = acc;
            }
            __syncthreads();
            if (t < 256) {
                // T_C = -T[32:64][32:64] Y2
                const int r = t >> 3, c4 = t & 7;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                float arow[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(Mm + (32 + r) * MLD + 32 + 4 * j);
                    arow[4 * j] = a4.x; arow[4 * j + 1] = a4.y; arow[4 * j + 2] = a4.z; arow[4 * j + 3] = a4.w;
                }
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const float a = arow[m];
                    const float4 yv = *reinterpret_cast<const float4 *>(Yt + m * 32 + 4 * c4);
                    acc.x = fmaf(a, yv.x, acc.x);
                    acc.y = fmaf(a, yv.y, acc.y);
                    acc.z = fmaf(a, yv.z, acc.z);
                    acc.w = fmaf(a, yv.w, acc.w);
                }
                *reinterpret_cast<float4 *>(Mm + (32 + r) * MLD + 4 * c4) =
                    make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
            }
            __syncthreads();
            // T' = (T - I) Diag(beta), bf16 K-major il [r][s] (B of U~ = T' V), and
            // -T Diag(beta), tf32 K-major il [r][s] (B of the W S term): one
            // 8-wide chunk of row r per thread
            {
                const int r = t >> 3, s0 = (t & 7) * 8;
                const float4 a = *reinterpret_cast<const float4 *>(Mm + r * MLD + s0);
                const float4 b4 = *reinterpret_cast<const float4 *>(Mm + r * MLD + s0 + 4);
                const float tv[8] = {a.x, a.y, a.z, a.w, b4.x, b4.y, b4.z, b4.w};
                float w8[8];
                uint32_t tb[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int s3 = s0 + u;
                    const float bs = s_beta[s3];
                    w8[u] = (s3 < r) ? tv[u] * bs : 0.f;
                    tb[u] = to_tf32(s3 < r ? -tv[u] * bs : (s3 == r ? -bs : 0.f));
                }
                *reinterpret_cast<uint4 *>(sm + SM_T + km_bf16(r, s0, 1024)) = pack_bf8(w8);
                *reinterpret_cast<uint4 *>(sm + SM_TB + km_tf32(r, s0, 2048)) = make_uint4(tb[0], tb[1], tb[2], tb[3]);
                *reinterpret_cast<uint4 *>(sm + SM_TB + km_tf32(r, s0 + 4, 2048)) = make_uint4(tb[4], tb[5], tb[6], tb[7]);
            }
        }
        fence_proxy_async_smem();
        sync_tc();

        // ===== M2: U = T' V - (T Diag(beta)) (K0 S)  (transposed) ============
        if (!wait_all(B.v, par)) { failed = true; break; }
        if (t == 0) {
            const uint32_t idv = instr_desc(kFmtBF16, 128, 64, 1, 0);
            const uint32_t idp = instr_desc(kFmtTF32, 128, 64, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = smem_desc(smem_u32(sm + SM_T + 256 * kk), 128, 1024, kSwizzleNone);
                const uint64_t av = smem_desc(smem_u32(sm + SM_STG_V + 2048 * kk), 8192, 1024, kSwizzle128B);
                mma_bf16_ss(tmem + TM_U, av, bd, idv, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bt = smem_desc(smem_u32(sm + SM_TB + 256 * kk), 128, 2048, kSwizzleNone);
                mma_tf32_ts(tmem + TM_U, tmem + TM_P + 8 * kk, bt, idp, 1);
            }
            mma_commit(B.mma);
        }
        if (!wait_all(B.mma, mma_phase)) { failed = true; break; }
        mma_phase ^= 1;
        tc_fence_after();

        // ===== E3: u = D_U + beta v, rounded to tf32 in place in TMEM ========
        float uv[16];
        {
            tmem_ld16(tmem + lane_base + TM_U + 16 * qt, uv);
            tmem_wait_ld();
            float ut[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int r = 16 * qt + k;
                uv[k] += s_beta[r] * bf(sm + SM_STG_V + sw_elem64(r, ch));
                ut[k] = __uint_as_float(to_tf32(uv[k]));
            }
            tmem_st16(tmem + lane_base + TM_U + 16 * qt, ut);
            tmem_wait_st();
        }
        sync_tc();

        // ===== M4: O += U^T A'^T;  dS = U^T Kbar (tf32, U^T read from TMEM) ===
        if (t == 0) {
            // v staging is consumed: load the next chunk's v
            if (ci + 1 < nchunks) issue_load_v(sm, &map_v, B.v, h, tok0 + c0 + C);
            const uint32_t ido = instr_desc(kFmtTF32, 128, 64, 0, 0);
            const uint32_t ids = instr_desc(kFmtTF32, 128, 128, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ba = smem_desc(smem_u32(sm + SM_A + 256 * kk), 128, 2048, kSwizzleNone);
                const uint64_t bk = smem_desc(smem_u32(sm + SM_KB + 256 * kk), 128, 2048, kSwizzleNone);
                mma_tf32_ts(tmem + TM_O, tmem + TM_U + 8 * kk, ba, ido, 1);
                mma_tf32_ts(tmem + TM_DS, tmem + TM_U + 8 * kk, bk, ids, kk > 0);
            }
            mma_commit(B.mma);
        }
        if (!wait_all(B.mma, mma_phase)) { failed = true; break; }
        mma_phase ^= 1;
        tc_fence_after();

        // ===== E4: o = D_O + (q.k) u;  S = e^{b_L} S + dS (TMEM) and bf16 copy
        {
            float ov[16];
            tmem_ld16(tmem + lane_base + TM_O + 16 * qt, ov);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int r = 16 * qt + k;
                if (r < Lc) o[((size_t)(tok0 + c0 + r) * H + h) * kDV + ch] = ov[k] + s_dq[r] * uv[k];
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const uint32_t col = 32 * qt + 16 * hh;
                float sv[16], dv[16];
                tmem_ld16(tmem + lane_base + TM_S + col, sv);
                tmem_ld16(tmem + lane_base + TM_DS + col, dv);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; ++c) sv[c] = fmaf(s_gam[col + c], sv[c], dv[c]);
                tmem_st16(tmem + lane_base + TM_S + col, sv);
#pragma unroll
                for (int c8 = 0; c8 < 2; ++c8) {
                    float x8[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) x8[u] = sv[8 * c8 + u];
                    *reinterpret_cast<uint4 *>(sm + SM_S + km_bf16(ch, col + 8 * c8, 2048)) = pack_bf8(x8);
                }
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        sync_tc();
    }

    asm volatile("cp.async.wait_all;" ::: "memory");
    if (failed) {
        if (t == 0) atomicOr(&g_kda_device_error, 1u);
        // let any copies or MMAs in flight finish (bounded) before freeing TMEM
        mbar_wait(B.mma, mma_phase, kWaitLimit);
        mbar_wait(B.qk, (uint32_t)(nchunks & 1) ^ 1u, kWaitLimit);
        mbar_wait(B.v, (uint32_t)(nchunks & 1) ^ 1u, kWaitLimit);
        mbar_wait(B.g, (uint32_t)(nchunks & 1) ^ 1u, kWaitLimit);
        __syncthreads();
    } else {
        // ---- final state: S_out[i][j] from the TMEM master (lane j, column i)
        float sv[32];
        tmem_ld32(tmem + lane_base + TM_S + 32 * qt, sv);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int i = 32 * qt + c;
            S_out[st_off + (size_t)i * kDV + ch] = sv[c];
        }
    }
    sync_tc();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, const float *S0, float *o, float *S_out,
                              const int32_t *cu_seqlens, int N, int64_t T, int H,
                              cudaStream_t stream) {
    CUtensorMap mq, mk, mv, mg;
    if (!make_map_bf16(&mq, q, T, H, 64, true) || !make_map_bf16(&mk, k, T, H, 64, true) ||
        !make_map_bf16(&mv, v, T, H, 64, true) || !make_map_f32(&mg, g, T, H))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)N * H;
    prefill_tc_kernel<<<(unsigned)blocks, NT, SMEM_ALLOC, stream>>>(mq, mk, mv, mg, g, beta, S0, o, S_out,
                                                                    cu_seqlens, N, H);
    return cudaGetLastError();
}

cudaError_t read_device_error(unsigned int *code, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_kda_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || !reset) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_kda_device_error, &zero, sizeof(unsigned int));
}

}  // namespace kda
