// prefill_tc.cu -- chunkwise prefill on Blackwell tensor cores (tcgen05), d = 128, C = 64.
//
// One CTA owns one (sequence, value head, 64-wide value tile) and walks the
// sequence's chunks in order, keeping its 128 x 64 slice of the state in fp32
// in tensor memory.  Every contraction of the chunk form ("You Could Have Come Up With
// Kimi Delta Attention", sec. 6.3-6.5; "From Attention to Learned Memory",
// sec. 4, WY/UT transform and the 16x16 blocked inverse) runs as a tcgen05 MMA
// with fp32 accumulators in tensor memory:
//
//   A-GEMM   [K+; Q+] K-^T               -> A_kk, A_qk                  M=128 N=64  K=128
//            (scalar decay: raw bf16 q, k, with the norms and exp(G_i - G_j)
//             applied to the result; per-channel decay: k^ exp(G - G_a),
//             q^ exp(G - G_a), k^ exp(G_a - G) of the normalised rows with a
//             mid-chunk anchor G_a, each split into bf16 high and low halves and
//             multiplied as hi*hi + hi*lo + lo*hi, ~16-bit precision over the
//             whole bf16 exponent range)
//   solve    T = (I + A_kk)^-1 on CUDA cores (16x16 forward substitution,
//            then T21 = -T22 A21 T11 merges), TB = T diag(beta)
//   X        [I; A_qk] TB          = [TB; A_qk TB]                    M=128 N=64  K=64
//   Y        [TB; A_qk TB] K~      = [W; A_qk W],  K~ = k exp(G)      M=128 N=128 K=64
//   chain    [TB, -W; A_qk TB, Q~ - A_qk W] [V; S]  = [E; O]          M=128 N=64  K=192
//            K_end^T E  = dS,  S <- diag(gamma) S + dS               M=128 N=64  K=64
//
// (E = U - W S are the corrected values and O = Q~ S + A_qk E the outputs of the
// chunk; folding A_qk into the first operand gives O from the same MMA as E.)
// Operands after the A-GEMM are fp16 (10-bit mantissa, the same as tf32).  The
// decayed keys and queries are bounded by 1 (unit rows, decay factors <= 1); v,
// E and the state must stay inside the fp16 range (|x| < 65504), which
// activations and states of normalised-key recurrences do.  The anchored
// per-channel factors exp(G_i - G_a), exp(G_a - G_j) need only stay finite in
// fp32 (cumulative decay below 80 nats over half a chunk, checked); outside
// these limits the fp32 CUDA-core path (KDA_FLAG_CUDA_CORES) is exact.
//
// The raw inputs of the next chunk are prefetched with cp.async into the
// staging buffers as soon as the current chunk no longer reads them, so their
// latency overlaps the chain MMAs.  Staging rows are padded so that threads
// owning different tokens read different banks.
//
// Shared-memory operands use the no-swizzle K-major core-matrix layout of
// tc_utils.cuh; the two operands written transposed by their producer threads
// (the state S^T and E^T) use a padded leading offset (144 B) to avoid bank
// conflicts.
#include "kda_common.cuh"
#include "prefill_plan.cuh"
#include "tc_utils.cuh"

namespace kda {

namespace tcp {

constexpr int C = 64;       // chunk
constexpr int D = 128;      // head size
constexpr int BV = 64;      // value columns per CTA
constexpr int NT = 256;     // threads (8 warps)
constexpr uint32_t kWaitLimit = 1u << 22;  // polls before a wait is declared stuck
constexpr float kMaxHalfChunkDecay = 80.0f;  // exp(80) stays finite in fp32 and bf16

// padded staging rows (elements)
constexpr int KS = D + 8;    // k, q rows: bf16, 272 B
constexpr int VS = BV + 8;   // v rows: bf16, 144 B
constexpr int GS = D + 4;    // G rows: fp32, 528 B

// shared-memory map (bytes)
constexpr uint32_t S_K = 0;                     // k staging bf16 [64][KS]
constexpr uint32_t S_Q = S_K + C * KS * 2;      // q staging bf16 [64][KS]
constexpr uint32_t S_V = S_Q + C * KS * 2;      // v staging bf16 [64][VS]
constexpr uint32_t S_G = S_V + C * VS * 2;      // per-channel log-decay -> exp(G - G_a), fp32 [64][GS]
constexpr uint32_t S_GS = S_G + C * GS * 4;     // scalar log-decay -> G [64]
constexpr uint32_t S_BETA = S_GS + 256;         // beta [64]
constexpr uint32_t S_RK = S_BETA + 256;         // 1/|k| [64]
constexpr uint32_t S_RQ = S_RK + 256;           // scale/|q| [64]
constexpr uint32_t S_EG = S_RQ + 256;           // scalar: exp(G_i) [64]
constexpr uint32_t S_EGL = S_EG + 256;          // scalar: exp(G_last - G_i) [64]
constexpr uint32_t S_GAM = S_EGL + 256;         // exp(G_last) [128]
constexpr uint32_t S_GA = S_GAM + 512;          // exp(G_a) at the anchor [128]
constexpr uint32_t S_EA = S_GA + 512;           // scalar: exp(G_i - G_a) [64]
constexpr uint32_t S_KF = S_EA + 256;           // scalar: exp(G_a - G_j) / |k_j| [64]
constexpr uint32_t R1 = (S_KF + 256 + 1023) & ~1023u;
//   A-GEMM operands, then the chain's first operands
constexpr uint32_t AK = R1;                    // [K+; Q+] 128 x 128 (16-bit)
constexpr uint32_t BK = AK + 128 * 128 * 2;    // K- 64 x 128
constexpr uint32_t A1 = R1;                    // [TB; A_qk TB] 128 x 64 fp16
constexpr uint32_t A2 = A1 + 128 * 64 * 2;     // [-W; Q~ - A_qk W] 128 x 128 fp16
constexpr uint32_t OST = R1;                   // o rows staged for coalesced stores, fp32 [64][OS]
constexpr int OS = BV + 4;                     // padded row (272 B)
constexpr uint32_t R2 = BK + 64 * 128 * 2;
//   triangular solve, then K~^T and K_end^T
constexpr int SP = 68;                         // padded, 16-byte aligned row of the fp32 solve tiles
constexpr uint32_t SOL_A = R2;                 // A_kk fp32 [64][SP]
constexpr uint32_t SOL_T = SOL_A + C * SP * 4; // T fp32 [64][SP]
constexpr uint32_t SOL_X = SOL_T + C * SP * 4; // merge temporaries fp32 [32][XP]
constexpr uint32_t KTT = R2;                   // K~^T 128 x 64 fp16
constexpr uint32_t KET = KTT + 128 * 64 * 2;   // K_end^T 128 x 64 fp16
constexpr int XP = 36;                         // row of the merge temporaries
constexpr uint32_t R3 = (SOL_X + 32 * XP * 4 + 127) & ~127u;
constexpr uint32_t LMAT = R3;                  // [I; A_qk] 128 x 64 fp16
constexpr uint32_t TBT = LMAT + 128 * 64 * 2;  // TB^T 64 x 64 fp16
constexpr uint32_t VT = TBT + 64 * 64 * 2;     // V^T 64 x 64 fp16
constexpr uint32_t ST = VT + 64 * 64 * 2;      // S^T 64 x 128 fp16, padded
constexpr uint32_t LBO_P = 144;                // padded leading byte offset
constexpr uint32_t ST_SBO = (D / 8) * LBO_P;
constexpr uint32_t ET = ST + (BV / 8) * ST_SBO;  // E^T 64 x 64 fp16, padded
constexpr uint32_t ET_SBO = (C / 8) * LBO_P;
constexpr uint32_t SMEM_BYTES = ET + (BV / 8) * ET_SBO;
static_assert(KET + 128 * 64 * 2 <= R3, "K~/K_end alias the solve area");
static_assert(A2 + 128 * 128 * 2 <= R2, "A1/A2 alias the A-GEMM operands");
static_assert(OST + C * OS * 4 <= R2, "o staging aliases the consumed chain operands");
static_assert(SMEM_BYTES + 64 <= 227 * 1024, "shared memory budget");
// per-channel decay: low bf16 halves of K- (A-GEMM B operand) live in the TB^T and V^T
// buffers, which are dead between a chunk's chain MMA and the next chunk's solve
constexpr uint32_t BKLO = TBT;
static_assert(VT == TBT + 64 * 64 * 2, "K- low half spans TB^T and V^T");

// TMEM columns
constexpr uint32_t T_A = 0, T_X = 64, T_Y = 128, T_D1 = 256, T_D2 = 320, T_ALO = 384,
                   T_S = 448, T_COLS = 512;

using tc::dense_sbo;
using tc::f16x8_store;
using tc::f16_bits;
using tc::bf16_at;
using tc::bf16x8_load;

}  // namespace tcp

// Issues the cp.async copies of one chunk's raw inputs into the staging buffers
// (rows past the sequence end are zero-filled).
template <bool PERCH>
__device__ __forceinline__ void tc_issue_loads(const Problem& P, unsigned char* smem, int64_t t0,
                                               int n, int kh, int h, int vt, int tid) {
  using namespace tcp;
  const int HV = P.HV;
  const uint32_t sbase = tc::smem_u32(smem);
  for (int u = tid; u < C * (D / 8); u += NT) {        // k, q: 16 pieces of 16 B per row
    const int i = u / (D / 8), q8 = u % (D / 8);
    const bool live = i < n;
    const int64_t t = live ? t0 + i : t0;
    const uint32_t nb = live ? 16u : 0u;
    tc::cp_async16(sbase + S_K + (i * KS + q8 * 8) * 2,
                   static_cast<const uint16_t*>(P.k) + t * P.k_stride + static_cast<int64_t>(kh) * D + q8 * 8, nb);
    tc::cp_async16(sbase + S_Q + (i * KS + q8 * 8) * 2,
                   static_cast<const uint16_t*>(P.q) + t * P.q_stride + static_cast<int64_t>(kh) * D + q8 * 8, nb);
  }
  for (int u = tid; u < C * (BV / 8); u += NT) {       // v: 8 pieces per row
    const int i = u / (BV / 8), q8 = u % (BV / 8);
    const bool live = i < n;
    const int64_t t = live ? t0 + i : t0;
    tc::cp_async16(sbase + S_V + (i * VS + q8 * 8) * 2,
                   static_cast<const uint16_t*>(P.v) + t * P.v_stride + static_cast<int64_t>(h) * D + vt * BV + q8 * 8,
                   live ? 16u : 0u);
  }
  if (PERCH) {
    for (int u = tid; u < C * (D / 4); u += NT) {      // g: 32 pieces per row
      const int i = u / (D / 4), q4 = u % (D / 4);
      const bool live = i < n;
      const int64_t t = live ? t0 + i : t0;
      tc::cp_async16(sbase + S_G + (i * GS + q4 * 4) * 4, P.g + (t * HV + h) * D + q4 * 4,
                     live ? 16u : 0u);
    }
  }
  if (tid < C) {
    const bool live = tid < n;
    const int64_t t = live ? t0 + tid : t0;
    tc::cp_async4(sbase + S_BETA + tid * 4, P.beta + t * HV + h, live ? 4u : 0u);
    if (!PERCH) tc::cp_async4(sbase + S_GS + tid * 4, P.g + t * HV + h, live ? 4u : 0u);
  }
  tc::cp_async_commit();
}

// DELTA = false is the additive write (no delta rule): a template parameter, so that the
// delta rule's code carries no test of it
template <bool PERCH, bool SBF16, bool DELTA>
__global__ void __launch_bounds__(tcp::NT, 1) tc_prefill_kernel(Problem P, PlanView plan) {
  using namespace tcp;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t s_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_anchored;     // scalar decay: anchored per-token factors are in range

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (plan.info[1] == 0) return;
  const int HV = P.HV;
  const SeqHeadTile cta = seq_head_tile(plan, HV, tcp::D / tcp::BV);
  const int b = cta.b, h = cta.h, vt = cta.vt;
  const int kh = h / (HV / P.HK);
  // additive write (no delta rule): A_kk = 0 makes T = I and K~ = 0 drops W = TB K~
  constexpr bool delta = DELTA;
  const uint32_t bos = P.offsets[b], eos = P.offsets[b + 1];
  // empty, or flagged by tc_range_scan_kernel: o and the slot are left as they were
  if (eos <= bos || plan.skip[static_cast<int64_t>(b) * HV + h] != 0) return;
  const int64_t sbase = (static_cast<int64_t>(P.slot_idx[b]) * HV + h) * D * D + vt * BV;

  float* sG = reinterpret_cast<float*>(smem + S_G);
  float* sGs = reinterpret_cast<float*>(smem + S_GS);
  float* sBeta = reinterpret_cast<float*>(smem + S_BETA);
  float* sRK = reinterpret_cast<float*>(smem + S_RK);
  float* sRQ = reinterpret_cast<float*>(smem + S_RQ);
  float* sEG = reinterpret_cast<float*>(smem + S_EG);
  float* sEGL = reinterpret_cast<float*>(smem + S_EGL);
  float* sGam = reinterpret_cast<float*>(smem + S_GAM);
  float* sGA = reinterpret_cast<float*>(smem + S_GA);
  float* sEA = reinterpret_cast<float*>(smem + S_EA);
  float* sKF = reinterpret_cast<float*>(smem + S_KF);
  float* sA = reinterpret_cast<float*>(smem + SOL_A);
  float* sT = reinterpret_cast<float*>(smem + SOL_T);
  float* sX = reinterpret_cast<float*>(smem + SOL_X);

  const uint32_t nchunks = (eos - bos + C - 1) / C;
  auto chunk_n = [&](uint32_t c) -> int {
    const int64_t t0 = static_cast<int64_t>(bos) + static_cast<int64_t>(c) * C;
    return static_cast<int>(min(static_cast<int64_t>(C), static_cast<int64_t>(eos) - t0));
  };
  tc_issue_loads<PERCH>(P, smem, bos, chunk_n(0), kh, h, vt, tid);

  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, T_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&s_bar, 1);
    tc::fence_mbar_init();
    s_abort = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  uint32_t phase = 0;

  // TMEM lane quarter of this warp and its column half
  const int row = 32 * (warp & 3) + lane;           // TMEM lane = M row
  const int chalf = warp >> 2;                      // 0 or 1
  const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;

  // the fp32 master state lives in tensor memory (lane = key channel `row`, columns
  // T_S + value column), so it costs no registers between chunk steps; its fp16 copy
  // S^T (N = value column j, K = key channel) is the chain MMA's B operand
  auto write_state_operand = [&](const float* Sv) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int jj = 32 * chalf + j;
      *reinterpret_cast<uint16_t*>(smem + ST + tc::cm_offset(jj, row, LBO_P, ST_SBO)) = f16_bits(Sv[j]);
    }
  };
  {
    const int64_t base = sbase + static_cast<int64_t>(row) * D + 32 * chalf;
    float Sv[32];
    uint32_t s0[16], s1[16];
    for (int j = 0; j < 32; ++j) {
      Sv[j] = SBF16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(P.pool)[base + j])
                    : static_cast<const float*>(P.pool)[base + j];
      if (j < 16) s0[j] = __float_as_uint(Sv[j]); else s1[j - 16] = __float_as_uint(Sv[j]);
    }
    tc::tmem_st16(tmem + lane_addr + T_S + 32 * chalf, s0);
    tc::tmem_st16(tmem + lane_addr + T_S + 32 * chalf + 16, s1);
    tc::tmem_wait_st();
    write_state_operand(Sv);
  }

  // the identity rows of L = [I; A_qk] never change
  if (row < C) {
    float idv[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) idv[e] = (32 * chalf + e == row) ? 1.f : 0.f;
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8)
      f16x8_store(smem, LMAT + tc::cm_offset(row, 32 * chalf + 8 * g8, 128, dense_sbo(64)),
                  idv + 8 * g8);
  }

  auto mma_wait = [&]() -> bool {
    const bool ok = tc::mbar_wait_bounded(&s_bar, phase & 1, kWaitLimit);
    phase ^= 1;
    if (!ok) s_abort = 1;
    tc::fence_after_sync();
    return ok;
  };

  for (uint32_t cidx = 0; cidx < nchunks; ++cidx) {
    const int64_t t0 = static_cast<int64_t>(bos) + static_cast<int64_t>(cidx) * C;
    const int n = chunk_n(cidx);

    // ---------------------------------------------------------------- phase 0: load
    tc::cp_async_wait_all();
    __syncthreads();

    // ---------------------------------------------------------------- phase 1: prep
    {                                                   // L2 norms: 4 threads per row
      // lanes l, l + 8, l + 16, l + 24 share row 8 warp + l, so that each 8-lane group of a
      // 16-byte shared-memory access reads 8 rows on different banks
      const int i = 8 * warp + (lane & 7), part = lane >> 3;
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        float kx[8], qx[8];
        bf16x8_load(smem + S_K + (i * KS + part * 32 + g8 * 8) * 2, kx);
        bf16x8_load(smem + S_Q + (i * KS + part * 32 + g8 * 8) * 2, qx);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sk += kx[e] * kx[e];
          sq += qx[e] * qx[e];
        }
      }
      sk += __shfl_xor_sync(0xffffffffu, sk, 8);
      sq += __shfl_xor_sync(0xffffffffu, sq, 8);
      sk += __shfl_xor_sync(0xffffffffu, sk, 16);
      sq += __shfl_xor_sync(0xffffffffu, sq, 16);
      if (part == 0) {
        sRK[i] = P.l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
        sRQ[i] = (P.l2norm ? rsqrtf(sq + 1e-6f) : 1.f) * P.scale;
      }
    }
    if (PERCH) {
      if (tid < D) {
        // channel tid: inclusive cumsum G, then E' = exp(G - G_a) in place, with the anchor
        // G_a at the chunk's middle token; exp(G_a) and exp(G_last) go to small arrays.
        // tc_range_scan_kernel has checked that G stays within kMaxHalfChunkDecay of G_a.
        float acc = 0.f;
#pragma unroll
        for (int i0 = 0; i0 < C; i0 += 16) {
          float gv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) gv[e] = sG[(i0 + e) * GS + tid];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            acc += gv[e];
            sG[(i0 + e) * GS + tid] = acc;
          }
        }
        const float ga = sG[((n - 1) / 2) * GS + tid];
#pragma unroll
        for (int i0 = 0; i0 < C; i0 += 16) {
          float gv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) gv[e] = sG[(i0 + e) * GS + tid];
#pragma unroll
          for (int e = 0; e < 16; ++e) sG[(i0 + e) * GS + tid] = __expf(gv[e] - ga);
        }
        sGam[tid] = __expf(acc);
        sGA[tid] = __expf(ga);
      }
    } else if (warp == 0) {                             // scalar: warp scan of 64 values
      const float g0 = sGs[2 * lane], g1 = sGs[2 * lane + 1];
      float s = g0 + g1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += y;
      }
      const float gl = __shfl_sync(0xffffffffu, s, 31);
      sGs[2 * lane] = s - g1;
      sGs[2 * lane + 1] = s;
      sEG[2 * lane] = __expf(s - g1);
      sEG[2 * lane + 1] = __expf(s);
      sEGL[2 * lane] = __expf(gl - (s - g1));
      sEGL[2 * lane + 1] = __expf(gl - s);
      const float gam = __expf(gl);
      sGam[lane] = gam; sGam[lane + 32] = gam; sGam[lane + 64] = gam; sGam[lane + 96] = gam;
      // anchored factors exp(G_i - G_a), exp(G_a - G_j) with the anchor mid-chunk, so that
      // exp(G_i - G_j) = product of two per-token values (used while both stay finite)
      const int am = (n - 1) / 2;
      const float ga = __shfl_sync(0xffffffffu, (am & 1) ? s : s - g1, am >> 1);
      const float d0 = (s - g1) - ga, d1 = s - ga;
      const bool ok = __all_sync(0xffffffffu, fmaxf(fabsf(d0), fabsf(d1)) <= kMaxHalfChunkDecay);
      sEA[2 * lane] = __expf(d0);
      sEA[2 * lane + 1] = __expf(d1);
      sKF[2 * lane] = __expf(-d0);
      sKF[2 * lane + 1] = __expf(-d1);
      if (lane == 0) s_anchored = ok ? 1 : 0;
    }
    __syncthreads();
    if (!PERCH && tid < C) sKF[tid] *= sRK[tid];
    // A-GEMM operands: [K+; Q+] (rows 0-63 keys, 64-127 queries) and K-.
    if (!PERCH) {
      // raw bf16 rows; consecutive threads fill one core matrix (8 rows x 16 B) at a time
      for (int u = tid; u < C * (D / 8); u += NT) {
        const int r = (u / (8 * (D / 8))) * 8 + (u & 7), q8 = (u >> 3) % (D / 8);
        const uint32_t ks = S_K + (r * KS + q8 * 8) * 2, qs = S_Q + (r * KS + q8 * 8) * 2;
        const uint4 kv = *reinterpret_cast<const uint4*>(smem + ks);
        *reinterpret_cast<uint4*>(smem + AK + tc::cm_offset(r, q8 * 8, 128, dense_sbo(D))) = kv;
        *reinterpret_cast<uint4*>(smem + BK + tc::cm_offset(r, q8 * 8, 128, dense_sbo(D))) = kv;
        *reinterpret_cast<uint4*>(smem + AK + tc::cm_offset(r + C, q8 * 8, 128, dense_sbo(D))) =
            *reinterpret_cast<const uint4*>(smem + qs);
      }
    } else {
      // normalised rows times exp(+-(G - G_a)), split into bf16 high and low halves
      // (x = hi + lo to about 16 bits with the full bf16 exponent range): the high halves
      // go to the shared-memory operands, the low half of [K+; Q+] to tensor memory
      {
        const int i = row < C ? row : row - C;
        const uint32_t src = (row < C ? S_K : S_Q) + (i * KS) * 2;
        const float rs = row < C ? sRK[i] : sRQ[i];
        uint32_t lo[32];
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
          const int cc = 64 * chalf + 8 * g8;
          float x[8];
          bf16x8_load(smem + src + cc * 2, x);
          const float4 g0 = *reinterpret_cast<const float4*>(sG + i * GS + cc);   // E'
          const float4 g1 = *reinterpret_cast<const float4*>(sG + i * GS + cc + 4);
          const float f[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          uint32_t hi[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float v0 = x[e] * rs * f[e], v1 = x[e + 1] * rs * f[e + 1];
            hi[e / 2] = tc::pack_bf16x2(v0, v1);
            const float h0 = __uint_as_float(hi[e / 2] << 16);
            const float h1 = __uint_as_float(hi[e / 2] & 0xffff0000u);
            lo[4 * g8 + e / 2] = tc::pack_bf16x2(v0 - h0, v1 - h1);
          }
          *reinterpret_cast<uint4*>(smem + AK + tc::cm_offset(row, cc, 128, dense_sbo(D))) =
              make_uint4(hi[0], hi[1], hi[2], hi[3]);
        }
        uint32_t l0[16], l1[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          l0[e] = lo[e];
          l1[e] = lo[16 + e];
        }
        tc::tmem_st16(tmem + lane_addr + T_ALO + 32 * chalf, l0);
        tc::tmem_st16(tmem + lane_addr + T_ALO + 32 * chalf + 16, l1);
        tc::tmem_wait_st();
      }
      {                                                   // K-: 4 threads per key row
        const int j = 8 * warp + (lane & 7), qq = lane >> 3;   // lanes 8 apart, as above
        const float rs = sRK[j];
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {
          const int cc = 32 * qq + 8 * g8;
          float x[8];
          bf16x8_load(smem + S_K + (j * KS + cc) * 2, x);
          const float4 g0 = *reinterpret_cast<const float4*>(sG + j * GS + cc);   // E'
          const float4 g1 = *reinterpret_cast<const float4*>(sG + j * GS + cc + 4);
          const float f[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float v0 = x[e] * rs * __fdividef(1.f, f[e]), v1 = x[e + 1] * rs * __fdividef(1.f, f[e + 1]);
            hi[e / 2] = tc::pack_bf16x2(v0, v1);
            const float h0 = __uint_as_float(hi[e / 2] << 16);
            const float h1 = __uint_as_float(hi[e / 2] & 0xffff0000u);
            lo[e / 2] = tc::pack_bf16x2(v0 - h0, v1 - h1);
          }
          *reinterpret_cast<uint4*>(smem + BK + tc::cm_offset(j, cc, 128, dense_sbo(D))) =
              make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(smem + BKLO + tc::cm_offset(j, cc, 128, dense_sbo(D))) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------------------------------------------------------- phase 2: A-GEMM
    if (tid == 0) {
      const uint32_t id = tc::idesc_f16(128, 64, tc::kBF16);
      for (int s = 0; s < D / 16; ++s)                   // hi x hi
        tc::mma_ss(tmem + T_A,
                   tc::smem_desc(tc::smem_u32(smem + AK) + s * 256, 128, dense_sbo(D)),
                   tc::smem_desc(tc::smem_u32(smem + BK) + s * 256, 128, dense_sbo(D)), id,
                   s > 0);
      if (PERCH) {
        for (int s = 0; s < D / 16; ++s)                 // hi x lo
          tc::mma_ss(tmem + T_A,
                     tc::smem_desc(tc::smem_u32(smem + AK) + s * 256, 128, dense_sbo(D)),
                     tc::smem_desc(tc::smem_u32(smem + BKLO) + s * 256, 128, dense_sbo(D)), id, 1);
        for (int s = 0; s < D / 16; ++s)                 // lo x hi (low half read from TMEM)
          tc::mma_ts(tmem + T_A, tmem + T_ALO + s * 8,
                     tc::smem_desc(tc::smem_u32(smem + BK) + s * 256, 128, dense_sbo(D)), id, 1);
      }
      tc::mma_commit(&s_bar);
    }
    mma_wait();

    // ---------------------------------------------------------------- phase 3: A_kk, A_qk
    {
      uint32_t r0[16], r1[16];
      tc::tmem_ld16(tmem + lane_addr + T_A + 32 * chalf, r0);
      tc::tmem_ld16(tmem + lane_addr + T_A + 32 * chalf + 16, r1);
      tc::tmem_wait_ld();
      const bool is_k = row < C;
      const int i = is_k ? row : row - C;
      // scalar decay multiplied raw bf16 rows: apply the norms, scale and exp(G_i - G_j)
      // here; per-channel decay multiplied normalised, decayed rows already
      const float ri = is_k ? (PERCH ? 1.f : sRK[i]) * sBeta[i] : (PERCH ? 1.f : sRQ[i]);
      float x[32];
      if (PERCH) {
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]) * ri;
      } else if (s_anchored) {                        // exp(G_i - G_j) = E_i F_j (anchored)
        const float rie = ri * sEA[i];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 kf = *reinterpret_cast<const float4*>(sKF + 32 * chalf + e);
          x[e] = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]) * rie * kf.x;
          x[e + 1] = __uint_as_float(e + 1 < 16 ? r0[e + 1] : r1[e - 15]) * rie * kf.y;
          x[e + 2] = __uint_as_float(e + 2 < 16 ? r0[e + 2] : r1[e - 14]) * rie * kf.z;
          x[e + 3] = __uint_as_float(e + 3 < 16 ? r0[e + 3] : r1[e - 13]) * rie * kf.w;
        }
      } else {                                        // exact per pair for extreme decays
        const float gi = sGs[i];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int j = 32 * chalf + e;
          x[e] = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]) * ri * sRK[j] * __expf(gi - sGs[j]);
        }
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int j = 32 * chalf + e;
        const bool keep = is_k ? (delta && j < i) : (j <= i);
        x[e] = keep ? x[e] : 0.f;
      }
      if (is_k) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(sA + i * SP + 32 * chalf + e) =
              make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
      } else {
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8)
          f16x8_store(smem, LMAT + tc::cm_offset(row, 32 * chalf + 8 * g8, 128, dense_sbo(64)),
                      x + 8 * g8);
      }
    }
    __syncthreads();

    // ---------------------------------------------------------------- phase 4: solve
    // the 32x32 merge reads the strictly-upper 16x16 blocks of T11 and T22: zero them
    for (int idx = tid; idx < 2 * 256; idx += NT) {
      const int blk = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
      sT[(32 * blk + r) * SP + 32 * blk + 16 + c] = 0.f;
    }
    // diagonal 16x16 blocks: lane (block, column) keeps its column of the block's inverse
    // in registers and substitutes row by row
    if (warp < 2) {
      const int base = (warp * 2 + (lane >> 4)) * 16, col = lane & 15;
      float t[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float v = r == col ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < r; ++m) v -= sA[(base + r) * SP + base + m] * t[m];
        t[r] = v;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) sT[(base + r) * SP + base + col] = t[r];
    }
    __syncthreads();
    // merges: T21 = -T22 (A21 T11), block size 16 (two pairs) then 32 (one pair);
    // each thread owns a 1 x 4 strip of the output
    if (tid < 128) {                                      // X = A21 T11, two 16x16 pairs
      const int p = tid >> 6, r = (tid >> 2) & 15, c = (tid & 3) * 4;
      const int r0 = 32 * p + 16, c0 = 32 * p;
      float a[16];
#pragma unroll
      for (int m = 0; m < 16; m += 4) {
        const float4 v = *reinterpret_cast<const float4*>(sA + (r0 + r) * SP + c0 + m);
        a[m] = v.x; a[m + 1] = v.y; a[m + 2] = v.z; a[m + 3] = v.w;
      }
      float4 t[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) t[m] = *reinterpret_cast<const float4*>(sT + (c0 + m) * SP + c0 + c);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        acc.x += a[m] * t[m].x; acc.y += a[m] * t[m].y; acc.z += a[m] * t[m].z; acc.w += a[m] * t[m].w;
      }
      *reinterpret_cast<float4*>(sX + (16 * p + r) * XP + c) = acc;
    }
    __syncthreads();
    if (tid < 128) {                                      // T21 = -T22 X
      const int p = tid >> 6, r = (tid >> 2) & 15, c = (tid & 3) * 4;
      const int r0 = 32 * p + 16, c0 = 32 * p;
      float a[16];
#pragma unroll
      for (int m = 0; m < 16; m += 4) {
        const float4 v = *reinterpret_cast<const float4*>(sT + (r0 + r) * SP + r0 + m);
        a[m] = v.x; a[m + 1] = v.y; a[m + 2] = v.z; a[m + 3] = v.w;
      }
      float4 x[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) x[m] = *reinterpret_cast<const float4*>(sX + (16 * p + m) * XP + c);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        acc.x += a[m] * x[m].x; acc.y += a[m] * x[m].y; acc.z += a[m] * x[m].z; acc.w += a[m] * x[m].w;
      }
      *reinterpret_cast<float4*>(sT + (r0 + r) * SP + c0 + c) =
          make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    __syncthreads();
    {                                                     // X = A21 T11, one 32x32 pair
      const int r = tid >> 3, c = (tid & 7) * 4;
      float a[32];                                        // row r of A21, loaded up front
#pragma unroll
      for (int m = 0; m < 32; m += 4) {
        const float4 v = *reinterpret_cast<const float4*>(sA + (32 + r) * SP + m);
        a[m] = v.x; a[m + 1] = v.y; a[m + 2] = v.z; a[m + 3] = v.w;
      }
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int m0 = 0; m0 < 32; m0 += 8) {
        float4 t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = *reinterpret_cast<const float4*>(sT + (m0 + e) * SP + c);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float av = a[m0 + e];
          acc.x += av * t[e].x; acc.y += av * t[e].y; acc.z += av * t[e].z; acc.w += av * t[e].w;
        }
      }
      *reinterpret_cast<float4*>(sX + r * XP + c) = acc;
    }
    __syncthreads();
    {                                                     // T21 = -T22 X
      const int r = tid >> 3, c = (tid & 7) * 4;
      float a[32];
#pragma unroll
      for (int m = 0; m < 32; m += 4) {
        const float4 v = *reinterpret_cast<const float4*>(sT + (32 + r) * SP + 32 + m);
        a[m] = v.x; a[m + 1] = v.y; a[m + 2] = v.z; a[m + 3] = v.w;
      }
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int m0 = 0; m0 < 32; m0 += 8) {
        float4 x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = *reinterpret_cast<const float4*>(sX + (m0 + e) * XP + c);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float av = a[m0 + e];
          acc.x += av * x[e].x; acc.y += av * x[e].y; acc.z += av * x[e].z; acc.w += av * x[e].w;
        }
      }
      *reinterpret_cast<float4*>(sT + (32 + r) * SP + c) =
          make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    __syncthreads();
    // TB^T[j][m] = T[m][j] beta_j  (N = j, K = m)
    for (int u = tid; u < C * (C / 8); u += NT) {
      const int j = u % C, m8 = u / C;
      const float bj = sBeta[j];
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {                      // T is lower triangular
        const int m = m8 * 8 + e;
        x[e] = m >= j ? sT[m * SP + j] * bj : 0.f;
      }
      f16x8_store(smem, TBT + tc::cm_offset(j, m8 * 8, 128, dense_sbo(64)), x);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------------------------------------------------------- phase 5: X
    if (tid == 0) {
      const uint32_t id = tc::idesc_f16(128, 64, tc::kF16);
      for (int s = 0; s < C / 16; ++s)
        tc::mma_ss(tmem + T_X,
                   tc::smem_desc(tc::smem_u32(smem + LMAT) + s * 256, 128, dense_sbo(64)),
                   tc::smem_desc(tc::smem_u32(smem + TBT) + s * 256, 128, dense_sbo(64)), id,
                   s > 0);
      tc::mma_commit(&s_bar);
    }
    // ---------------------------------------------------------------- phase 6: K~^T, K_end^T, V^T
    for (int u = tid; u < D * (C / 8); u += NT) {         // (channel c, 8 tokens)
      const int c = u % D, m8 = u / D;
      float kt[8], ke[8];
      if (PERCH) {
        const float El = sG[(C - 1) * GS + c], ea = sGA[c];   // E'_last, exp(G_a)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int m = m8 * 8 + e;
          const float Em = sG[m * GS + c];
          const float kx = bf16_at(smem, S_K, m * KS + c) * sRK[m];
          kt[e] = delta ? kx * Em * ea : 0.f;                // k^ exp(G_m)
          ke[e] = kx * __fdividef(El, Em);                   // k^ exp(G_last - G_m)
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int m = m8 * 8 + e;
          const float kx = bf16_at(smem, S_K, m * KS + c) * sRK[m];
          kt[e] = delta ? kx * sEG[m] : 0.f;
          ke[e] = kx * sEGL[m];
        }
      }
      f16x8_store(smem, KTT + tc::cm_offset(c, m8 * 8, 128, dense_sbo(64)), kt);
      f16x8_store(smem, KET + tc::cm_offset(c, m8 * 8, 128, dense_sbo(64)), ke);
    }
    for (int u = tid; u < BV * (C / 8); u += NT) {        // (value column j, 8 tokens)
      const int j = u % BV, m8 = u / BV;
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = bf16_at(smem, S_V, (m8 * 8 + e) * VS + j);
      f16x8_store(smem, VT + tc::cm_offset(j, m8 * 8, 128, dense_sbo(64)), x);
    }
    tc::fence_async_smem();
    mma_wait();

    // ---------------------------------------------------------------- phase 7: A1 = X
    {
      uint32_t r0[16], r1[16];
      tc::tmem_ld16(tmem + lane_addr + T_X + 32 * chalf, r0);
      tc::tmem_ld16(tmem + lane_addr + T_X + 32 * chalf + 16, r1);
      tc::tmem_wait_ld();
      float x[32];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        x[e] = __uint_as_float(r0[e]);
        x[e + 16] = __uint_as_float(r1[e]);
      }
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        f16x8_store(smem, A1 + tc::cm_offset(row, 32 * chalf + 8 * g8, 128, dense_sbo(64)),
                    x + 8 * g8);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------------------------------------------------------- phase 8: Y
    if (tid == 0) {
      const uint32_t id = tc::idesc_f16(128, 128, tc::kF16);
      for (int s = 0; s < C / 16; ++s)
        tc::mma_ss(tmem + T_Y,
                   tc::smem_desc(tc::smem_u32(smem + A1) + s * 256, 128, dense_sbo(64)),
                   tc::smem_desc(tc::smem_u32(smem + KTT) + s * 256, 128, dense_sbo(64)), id,
                   s > 0);
      tc::mma_commit(&s_bar);
    }
    mma_wait();

    // ---------------------------------------------------------------- phase 9: A2
    uint32_t ry[2][32];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t a[16], b[16];
      tc::tmem_ld16(tmem + lane_addr + T_Y + 64 * chalf + 32 * half, a);
      tc::tmem_ld16(tmem + lane_addr + T_Y + 64 * chalf + 32 * half + 16, b);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        ry[half][e] = a[e];
        ry[half][e + 16] = b[e];
      }
    }
    tc::tmem_wait_ld();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int c0 = 64 * chalf + 32 * half;
      float x[32];
      if (row >= C) {                                     // Q~ = q scale/|q| exp(G)
        const int i = row - C;
        const float rq = sRQ[i];
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {
          float qv[8];
          bf16x8_load(smem + S_Q + (i * KS + c0 + 8 * g8) * 2, qv);
          if (PERCH) {
            const float4 ga = *reinterpret_cast<const float4*>(sG + i * GS + c0 + 8 * g8);
            const float4 gb = *reinterpret_cast<const float4*>(sG + i * GS + c0 + 8 * g8 + 4);
            const float4 aa = *reinterpret_cast<const float4*>(sGA + c0 + 8 * g8);
            const float4 ab = *reinterpret_cast<const float4*>(sGA + c0 + 8 * g8 + 4);
            const float gv[8] = {ga.x * aa.x, ga.y * aa.y, ga.z * aa.z, ga.w * aa.w,
                                 gb.x * ab.x, gb.y * ab.y, gb.z * ab.z, gb.w * ab.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) x[8 * g8 + e] = qv[e] * rq * gv[e];   // exp(G_i)
          } else {
            const float f = rq * sEG[i];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[8 * g8 + e] = qv[e] * f;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) x[e] -= __uint_as_float(ry[half][e]);
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        f16x8_store(smem, A2 + tc::cm_offset(row, c0 + 8 * g8, 128, dense_sbo(D)), x + 8 * g8);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // the staging buffers are free: prefetch the next chunk's inputs
    if (cidx + 1 < nchunks)
      tc_issue_loads<PERCH>(P, smem, t0 + C, chunk_n(cidx + 1), kh, h, vt, tid);

    // ---------------------------------------------------------------- phase 10: [E; O]
    if (tid == 0) {
      const uint32_t id = tc::idesc_f16(128, BV, tc::kF16);
      for (int s = 0; s < C / 16; ++s)     // [TB; A_qk TB] V
        tc::mma_ss(tmem + T_D1,
                   tc::smem_desc(tc::smem_u32(smem + A1) + s * 256, 128, dense_sbo(64)),
                   tc::smem_desc(tc::smem_u32(smem + VT) + s * 256, 128, dense_sbo(64)), id,
                   s > 0);
      for (int s = 0; s < D / 16; ++s)     // [-W; Q~ - A_qk W] S
        tc::mma_ss(tmem + T_D1,
                   tc::smem_desc(tc::smem_u32(smem + A2) + s * 256, 128, dense_sbo(D)),
                   tc::smem_desc(tc::smem_u32(smem + ST) + s * 2 * LBO_P, LBO_P, ST_SBO), id, 1);
      tc::mma_commit(&s_bar);
    }
    mma_wait();

    // ---------------------------------------------------------------- phase 11: E^T, o
    {
      uint32_t r0[16], r1[16];
      tc::tmem_ld16(tmem + lane_addr + T_D1 + 32 * chalf, r0);
      tc::tmem_ld16(tmem + lane_addr + T_D1 + 32 * chalf + 16, r1);
      tc::tmem_wait_ld();
      if (row < C) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float ev = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]);
          *reinterpret_cast<uint16_t*>(smem + ET + tc::cm_offset(32 * chalf + e, row, LBO_P, ET_SBO)) =
              f16_bits(ev);
        }
      } else {
        // o rows go through shared memory (the chain operands there are consumed) so
        // that the global stores below are coalesced
        float* op = reinterpret_cast<float*>(smem + OST) + (row - C) * OS + 32 * chalf;
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          *reinterpret_cast<float4*>(op + e) =
              make_float4(__uint_as_float(r0[e]), __uint_as_float(r0[e + 1]),
                          __uint_as_float(r0[e + 2]), __uint_as_float(r0[e + 3]));
          *reinterpret_cast<float4*>(op + 16 + e) =
              make_float4(__uint_as_float(r1[e]), __uint_as_float(r1[e + 1]),
                          __uint_as_float(r1[e + 2]), __uint_as_float(r1[e + 3]));
        }
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // coalesced o stores: each warp instruction writes two whole 256-byte token rows
#pragma unroll
    for (int k = 0; k < (C * BV / 4) / NT; ++k) {
      const int idx = tid + k * NT, i = idx / (BV / 4), q = idx % (BV / 4);
      if (i < n)
        *reinterpret_cast<float4*>(P.o + ((t0 + i) * HV + h) * D + vt * BV + q * 4) =
            *reinterpret_cast<const float4*>(smem + OST + (i * OS + q * 4) * 4);
    }

    // ---------------------------------------------------------------- phase 12: dS
    if (tid == 0) {
      const uint32_t id = tc::idesc_f16(128, BV, tc::kF16);
      for (int s = 0; s < C / 16; ++s)
        tc::mma_ss(tmem + T_D2,
                   tc::smem_desc(tc::smem_u32(smem + KET) + s * 256, 128, dense_sbo(64)),
                   tc::smem_desc(tc::smem_u32(smem + ET) + s * 2 * LBO_P, LBO_P, ET_SBO), id,
                   s > 0);
      tc::mma_commit(&s_bar);
    }
    mma_wait();

    // ---------------------------------------------------------------- phase 13: S update
    {
      uint32_t r0[16], r1[16], s0[16], s1[16];
      tc::tmem_ld16(tmem + lane_addr + T_D2 + 32 * chalf, r0);
      tc::tmem_ld16(tmem + lane_addr + T_D2 + 32 * chalf + 16, r1);
      tc::tmem_ld16(tmem + lane_addr + T_S + 32 * chalf, s0);
      tc::tmem_ld16(tmem + lane_addr + T_S + 32 * chalf + 16, s1);
      tc::tmem_wait_ld();
      const float gam = sGam[row];
      float Sv[32];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        Sv[e] = gam * __uint_as_float(s0[e]) + __uint_as_float(r0[e]);
        Sv[e + 16] = gam * __uint_as_float(s1[e]) + __uint_as_float(r1[e]);
        s0[e] = __float_as_uint(Sv[e]);
        s1[e] = __float_as_uint(Sv[e + 16]);
      }
      tc::tmem_st16(tmem + lane_addr + T_S + 32 * chalf, s0);
      tc::tmem_st16(tmem + lane_addr + T_S + 32 * chalf + 16, s1);
      tc::tmem_wait_st();
      write_state_operand(Sv);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (s_abort) break;
  }
  tc::cp_async_wait_all();

  if (s_abort) {
    // give the tensor core a last bounded chance to drain before TMEM is released
    tc::mbar_wait_bounded(&s_bar, phase & 1, kWaitLimit);
    if (tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
  } else {
    const int64_t base = sbase + static_cast<int64_t>(row) * D + 32 * chalf;
    uint32_t s0[16], s1[16];
    tc::tmem_ld16(tmem + lane_addr + T_S + 32 * chalf, s0);
    tc::tmem_ld16(tmem + lane_addr + T_S + 32 * chalf + 16, s1);
    tc::tmem_wait_ld();
    for (int j = 0; j < 32; ++j) {
      const float v = __uint_as_float(j < 16 ? s0[j] : s1[j - 16]);
      if (SBF16)
        static_cast<uint16_t*>(P.pool)[base + j] = f32_to_bf16_bits(v);
      else
        static_cast<float*>(P.pool)[base + j] = v;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, T_COLS);
}

// The per-channel factors exp(G_i - G_a), exp(G_a - G_j) of the kernel above (anchor G_a at
// a chunk's middle token) must stay finite in fp32, which bounds how far a channel's
// cumulative log-decay may move from the anchor within a chunk.  The kernel walks a
// sequence's chunks in order and writes o as it goes, so it cannot find a chunk outside
// that range before it has written the earlier ones.  This pass checks every chunk first
// (the same cumulative sums, in the same order, against a bound one nat tighter) and marks
// the (sequence, head) of a chunk outside it: the kernel then leaves its o rows and its slot
// untouched, and the device error word reports KDA_DEVERR_DECAY_RANGE.
constexpr float kScanHalfChunkDecay = tcp::kMaxHalfChunkDecay - 1.0f;

__global__ void __launch_bounds__(tcp::D) tc_range_scan_kernel(Problem P, PlanView plan) {
  using namespace tcp;
  const int gc = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int plan_valid = plan.info[1], plan_chunks = plan.info[0];
  const ChunkInfo ci = plan.chunks[gc];
  if (plan_valid == 0 || gc >= plan_chunks) return;
  const int HV = P.HV, am = (ci.n - 1) / 2;
  const float* g = P.g + (ci.t0 * HV + h) * D + c;
  float acc = 0.f, gmin = 0.f, gmax = -3.0e38f, ga = 0.f;
#pragma unroll 16
  for (int i = 0; i < C; ++i) {
    acc += i < ci.n ? g[static_cast<int64_t>(i) * HV * D] : 0.f;
    gmin = fminf(gmin, acc);
    gmax = fmaxf(gmax, acc);
    ga = i == am ? acc : ga;
  }
  if (__syncthreads_or(fmaxf(gmax - ga, ga - gmin) > kScanHalfChunkDecay) && c == 0) {
    plan.skip[static_cast<int64_t>(ci.seq) * HV + h] = 1;
    raise_device_error(P.err, KDA_DEVERR_DECAY_RANGE);
  }
}

bool tc_prefill_supported(const Problem& P, bool qbf16) {
  return qbf16 && P.D == tcp::D && P.chunk == tcp::C;
}

size_t tc_workspace_bytes(const Problem& P) { return plan_layout(P, nullptr, 0, nullptr); }

template <bool PERCH, bool SBF16>
static cudaError_t launch_tc_t(const Problem& P, const PlanView& plan, cudaStream_t st) {
  auto k = (P.flags & KDA_FLAG_NO_DELTA) ? tc_prefill_kernel<PERCH, SBF16, false>
                                         : tc_prefill_kernel<PERCH, SBF16, true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(tcp::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  const unsigned ctas = seq_head_tile_ctas(P, tcp::D / tcp::BV);
  if (ctas == 0) return cudaErrorInvalidConfiguration;
  k<<<ctas, tcp::NT, tcp::SMEM_BYTES, st>>>(P, plan);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const Problem& P, void* workspace, bool perch, bool sbf16,
                              cudaStream_t stream, const Stages& st) {
  PlanView plan;
  plan_layout(P, static_cast<char*>(workspace), 0, &plan);
  st.mark(0, stream);
  cudaError_t e = launch_plan(P, plan, stream);
  if (e != cudaSuccess) return e;
  st.mark(1, stream);
  int k = 2;
  if (perch) {
    tc_range_scan_kernel<<<dim3(static_cast<unsigned>(plan_max_chunks(P)), P.HV), tcp::D, 0, stream>>>(P, plan);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    st.mark(k++, stream);
    e = sbf16 ? launch_tc_t<true, true>(P, plan, stream) : launch_tc_t<true, false>(P, plan, stream);
  } else {
    e = sbf16 ? launch_tc_t<false, true>(P, plan, stream) : launch_tc_t<false, false>(P, plan, stream);
  }
  st.mark(k, stream);
  return e;
}

}  // namespace kda
