// prefill_split.cu -- chunkwise prefill on Blackwell tensor cores in two kernels:
// a chunk-parallel front kernel and a sequential chain kernel (d = 128, C = 64).
//
// The chunk form ("You Could Have Come Up With Kimi Delta Attention", sec. 6.3-6.5;
// "From Attention to Learned Memory", sec. 4, WY/UT transform) splits every chunk's
// work into a part that depends only on the chunk's own keys, queries, gates and
// betas -- the intra-chunk matrices A_kk and A_qk, the inverse T = (I + A_kk)^-1 and
// the WY factors -- and a part that carries the state from chunk to chunk.  With
// E = TB V - W S = TB (V - K~ S) the chunk's corrections (W = TB K~), the state update and
// the output are
//
//   S' = diag(gam) S + K_end^T E = diag(gam) S + Kb E',   Kb = K_end^T TB,  E' = V - K~ S
//   O  = Q~ S + A_qk E           = Q~ S + A1o E',         A1o = A_qk TB
//
// so every product that does not involve the state can be formed before the state is
// known.  The front kernel runs one CTA per (chunk, value head) over the whole GPU and
// writes each chunk's operands to the workspace:
//
//   Kb          128 x 64    fp16   (rows = key channels)
//   [K~; Q~]    128 x 128   fp16   (rows = tokens; K = key channels)
//   A1o          64 x 64    fp16
//   gam = exp(G_last) per key channel, fp32
//
// Kb is stored per thread of the chain kernel (each thread's 16-byte pieces of its row,
// interleaved across threads so that every warp access is contiguous): the chain kernel
// loads it into registers and writes it to tensor memory, where the MMA reads its A
// operand.  [K~; Q~] and A1o are stored in the K-major core-matrix order of shared-memory
// A operands and moved with one bulk copy.  The chain kernel keeps a (sequence, value
// head, 64 value columns) slice of the state in registers; per chunk two dependent MMA
// groups are on the sequential path,
//
//   X = [K~; Q~] S                M=128 N=64 K=128     (rows 0-63 K~ S, rows 64-127 Q~ S)
//   E' = V - X[0:64]              (fp16, over V in shared memory)
//   D = Kb E'                     M=128 N=64 K=64      (A from tensor memory)
//   S <- diag(gam) S + D
//
// and the output MMA A1o E' accumulates onto rows 64-127 of X beside the state update.
// Every operand the threads produce (V, E', S, and in the front kernel TB and K_end) is
// stored MN-major, so each thread writes whole 16-byte rows of core matrices instead of
// transposing.  Against a record holding P = -Kb K~ (128 x 128) and A2o = Q~ - A1o K~ in
// place of [K~; Q~], this one is 22% smaller and the front kernel runs one MMA round fewer,
// at the cost of a second dependent MMA on the chain's sequential path.
//
// Operand precisions are those of the single-kernel path in prefill_tc.cu (fp16 operands,
// fp32 accumulation and fp32 state); the state passes through fp16 as the B operand of
// [K~; Q~] S, and E' as that of Kb E' and A1o E'.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "prefill_plan.cuh"
#include "tc_utils.cuh"

namespace kda {

namespace tcs {

constexpr int C = 64;       // chunk
constexpr int D = 128;      // head size
constexpr int BV = 64;      // value columns per chain CTA
constexpr int NT = 256;     // threads (8 warps); the chain kernel's compute warps
constexpr int NTD = 128;    // chain kernel: operand warps 8-11
constexpr int NTO = 64;     // chain kernel: output warps 14-15 (TMEM lanes 64-127)
constexpr int NTC = NT + NTD + 64 + NTO;   // + warp 12, whose lane 0 issues the output MMA,
                                           // and warp 13, which only pads to warp 14
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kMaxHalfChunkDecay = 80.0f;

// record of one (chunk, value head) in the workspace
//   BLOB: piece p (0..3) of thread t at (p * NT + t) * 16; thread t (key channel
//         r = 32 (warp & 3) + lane, column half h = warp >> 2) holds Kb[r][32h .. 32h+32)
//   KQ:   [K~; Q~] (rows 0-63 K~, rows 64-127 Q~, K = key channel), element (row, channel c)
//         at cm_offset(row, c, 128, KQ_SBO): the K-major A operand of [K~; Q~] S
//   A1O:  A1o (token m, column j) at cm_offset(m, j, 128, A1O_SBO), right after KQ, so that
//         KQ and A1O move with one bulk copy
//   GAM:  exp(G_last) per key channel
constexpr uint32_t BLOB_PIECES = 4;
constexpr uint32_t REC_BLOB = 0;
constexpr uint32_t REC_KQ = REC_BLOB + BLOB_PIECES * 256 * 16;
constexpr uint32_t KQ_SBO = tc::dense_sbo(D), KQ_BYTES = 2 * C * D * 2;
constexpr uint32_t REC_A1O = REC_KQ + KQ_BYTES;
constexpr uint32_t A1O_SBO = tc::dense_sbo(C), A1O_BYTES = C * C * 2;
constexpr uint32_t KQA_BYTES = KQ_BYTES + A1O_BYTES;   // one bulk copy
constexpr uint32_t REC_GAM = REC_A1O + A1O_BYTES;
constexpr uint32_t REC_BYTES = REC_GAM + 128 * 4;    // 57856, a multiple of 16
constexpr uint32_t KE_LBO = 2048, KE_SBO = 128;      // K_end (M = channel, K = token), MN-major
constexpr uint32_t TB_LBO = 1024, TB_SBO = 128;      // TB (N = column j, K = row m)
static_assert(REC_BYTES % 16 == 0 && REC_KQ % 16 == 0 && KQA_BYTES % 16 == 0,
              "records must stay 16-byte aligned");

// per-chunk vectors of the front kernel (byte offsets inside its SMALL area)
constexpr uint32_t O_GS = 0, O_BETA = 256, O_RK = 512, O_RQ = 768, O_EG = 1024, O_EGL = 1280,
                   O_GAM = 1536, O_GA = 2048, O_EA = 2560, O_KF = 2816, O_EL = 3072,
                   SMALL_BYTES = 3584;

// the fp32 solve tiles (A_kk and T, 64 x 64): element (r, c) at sidx(r, c), whose 4-float
// groups are permuted by r % 8 so that column-wise and row-wise 16-byte accesses both
// spread over the banks; a 16-byte group from c % 4 == 0 stays contiguous
__device__ __forceinline__ int sidx(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }
constexpr int SOL_TILE = 64 * 64 * 4;

// float index of element (token m, channel c) of the staged per-channel log-decay: four
// quarters of 32 channels, 64 rows of 128 bytes each, 16-byte chunks swizzled by m % 8
// (the TMA copies' 128-byte swizzle); 4 consecutive channels from c % 4 == 0 stay adjacent
__device__ __forceinline__ int g_off(int m, int c) {
  return (c >> 5) * (64 * 32) + m * 32 + ((((c & 31) >> 2) ^ (m & 7)) << 2) + (c & 3);
}
constexpr int XP = 36;      // row of the merge temporaries
constexpr uint32_t SOL_BYTES = 2 * SOL_TILE + 32 * XP * 4;

template <bool PERCH>
struct FrontMap;

// Scalar decay: four TMA copies put the raw k and q rows straight into the A-GEMM
// operand [K; Q], K-major in the 128-byte swizzled layout: two halves of 64 channels,
// each 128 rows (k rows 0-63, q rows 64-127) of 128 bytes; the key rows double as the
// B operand.
template <>
struct FrontMap<false> {
  static constexpr uint32_t AK = 0, AK_HALF = 128 * 128;
  static constexpr uint32_t SMALL = AK + 2 * AK_HALF;
  static constexpr uint32_t R2 = SMALL + SMALL_BYTES;   // solve, then K_end
  static constexpr uint32_t LMAT = R2 + SOL_BYTES;      // [*; A_qk] 128 x 64 fp16
  static constexpr uint32_t TBT = LMAT + 128 * 64 * 2;  // TB 64 x 64 fp16, MN-major
  static constexpr uint32_t BYTES = TBT + 64 * 64 * 2;
  static constexpr uint32_t KEA = R2;                   // K_end (MN-major)
};

// Per-channel decay: TMA copies stage the raw k and q rows (the 128-byte swizzled layout
// of the scalar path) and the log-decay rows (four 32-channel quarters, each 64 rows of
// 128 bytes, swizzled the same way).  The A-GEMM operands are the normalised, decayed rows
// as split bf16: [K+; Q+] high halves overwrite the raw rows in place, its low halves go to
// tensor memory, K- (both halves) to BK | BKLO.  Once the A-GEMM is done, K~ and Q~ are
// rebuilt from the two halves of [K+; Q+] and K_end from K-, so the staged rows, the
// log-decay and K- can all be reused: every region below serves several phases, which keeps
// two CTAs per SM.  K~ and Q~ go straight to the record.
template <>
struct FrontMap<true> {
  static constexpr uint32_t AK_HALF = 128 * 128;
  static constexpr uint32_t RAW = 0;                    // raw k | q -> [K+; Q+] high halves;
                                                        // then TB (half 0 k rows), A_qk (half 1
                                                        // k rows), Q~ in place (q rows)
  static constexpr uint32_t S_G = RAW + 2 * AK_HALF;    // log-decay -> exp(G - G_a); then K_end
  static constexpr uint32_t SMALL = S_G + C * D * 4;
  static constexpr uint32_t BK = SMALL + SMALL_BYTES;   // K- high | low halves; then the solve
  static constexpr uint32_t BKLO = BK + 64 * 128 * 2;   // tiles
  static constexpr uint32_t R2 = BK;
  static constexpr uint32_t BYTES = R2 + SOL_BYTES;
  static constexpr uint32_t TBT = RAW;
  static constexpr uint32_t LMAT = RAW + AK_HALF - 64 * 64 * 2;   // rows 64-127: half 1 k rows
  static constexpr uint32_t KEA = S_G;
  static_assert(R2 + 2 * SOL_TILE == BKLO + 64 * 128 * 2, "solve tiles cover the K- halves");
};

// front TMEM columns: A_kk/A_qk (second issuer's half of K in F_X), then Kb | A1o; the low
// half of [K+; Q+] in F_ALO
constexpr uint32_t F_A = 0, F_X = 64, F_ALO = 128, F_COLS = 256;

// chain shared memory (MN-major operands: core matrices of 8 K-rows x 8 value columns,
// value-column groups adjacent, K groups 1024 bytes apart).  A slot of the KQA ring holds a
// record's [K~; Q~ | A1o] as one bulk copy moves it; a V slot holds V, then E' = V - K~ S in
// place.  The output MMA A1o E' has M = 128 with A1o as rows 64-127: its A operand starts
// A1O_BYTES before A1o, so that rows 0-63 read the tail of Q~, whose products land in
// accumulator rows that are never read again.
constexpr uint32_t OP_LBO = 1024, OP_SBO = 128;
constexpr int OS = BV + 4;                               // o staging row (fp32)
constexpr uint32_t KQA_SLOTS = 3, V_SLOTS = 5;
constexpr uint32_t V_BYTES = 64 * 64 * 2, S_BYTES = 128 * 64 * 2;
constexpr uint32_t CH_KQA = 0;                           // [K~; Q~ | A1o] of three chunks
constexpr uint32_t CH_V = CH_KQA + KQA_SLOTS * KQA_BYTES;   // V -> E' of five chunks, 64 x 64 fp16
constexpr uint32_t CH_ST = CH_V + V_SLOTS * V_BYTES;     // S, 128 x 64 fp16
constexpr uint32_t CH_OST = CH_ST + S_BYTES;             // o rows fp32 [64][OS]
constexpr uint32_t CH_GAM = CH_OST + C * OS * 4;         // gamma of four chunks, fp32 [4][128]
constexpr uint32_t GAM_SLOTS = 4;
constexpr uint32_t CH_BYTES = CH_GAM + GAM_SLOTS * D * 4;
static_assert(CH_BYTES + 64 <= 227 * 1024, "chain shared memory budget");
static_assert(2 * (FrontMap<true>::BYTES + 3 * 1024) <= 228 * 1024, "two per-channel front CTAs per SM");
static_assert(2 * (FrontMap<false>::BYTES + 1024 + 1024) <= 228 * 1024, "two scalar front CTAs per SM");
static_assert(CH_V % 128 == 0 && CH_ST % 128 == 0 && KQA_BYTES % 128 == 0, "operand alignment");
// chain TMEM columns: Kb of two chunks (fp16 pairs); the state MMA Kb E' as two partial
// sums (one per issuing thread); [K~; Q~] S as two partial sums, double-buffered (rows 0-63
// K~ S, rows 64-127 Q~ S, onto which A1o E' accumulates the output)
constexpr uint32_t T_A = 0, A_COLS = 32, T_DS = 64, T_DS2 = 128, T_X = 192, CH_COLS = 512;
__host__ __device__ constexpr uint32_t x_col(uint32_t c, uint32_t part) {
  return T_X + (c & 1) * 128 + part * 64;
}
static_assert(x_col(1, 1) + 64 <= CH_COLS, "chain tensor-memory columns");

__device__ __forceinline__ uint4 f16x8_pack(const float* x) {
  return make_uint4(tc::pack_f16x2(x[0], x[1]), tc::pack_f16x2(x[2], x[3]),
                    tc::pack_f16x2(x[4], x[5]), tc::pack_f16x2(x[6], x[7]));
}

}  // namespace tcs

// cp.async copies of one chunk's beta and, for scalar decay, log-decay (rows past n
// zero-filled); k, q and a per-channel log-decay come by TMA
template <bool PERCH>
__device__ __forceinline__ void front_issue_loads(const Problem& P, unsigned char* smem,
                                                  int64_t t0, int n, int kh, int h, int tid) {
  using namespace tcs;
  using M = FrontMap<PERCH>;
  const int HV = P.HV;
  const uint32_t sb = tc::smem_u32(smem);
  if (tid < C) {
    const bool live = tid < n;
    const int64_t t = live ? t0 + tid : t0;
    tc::cp_async4(sb + M::SMALL + O_BETA + tid * 4, P.beta + t * HV + h, live ? 4u : 0u);
    if (!PERCH) tc::cp_async4(sb + M::SMALL + O_GS + tid * 4, P.g + t * HV + h, live ? 4u : 0u);
  }
  tc::cp_async_commit();
}

// One CTA per (chunk, value head): everything of the chunk that does not depend on the
// state, written to the chunk's record.
// DELTA = false is the additive write (no delta rule): A_kk = 0 makes T = I and K~ = 0
// drops W = TB K~; a template parameter, so that the delta rule's code carries no test of it
template <bool PERCH, bool DELTA>
__global__ void __launch_bounds__(tcs::NT, 2)
    tc_front_kernel(Problem P, PlanView plan, unsigned char* records,
                    const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmg) {
  using namespace tcs;
  using M = FrontMap<PERCH>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzled operand needs a 1024-byte aligned base; the launch adds 1 KB of slack
  unsigned char* const smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t s_bar;                    // MMAs issued by thread 0
  __shared__ uint64_t s_bar2;                   // MMAs issued by thread 32
  __shared__ uint64_t s_ld;                     // TMA copies of k and q (scalar decay)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_range;
  __shared__ int s_anchored;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gc = blockIdx.x, h = blockIdx.y;
  // the three table reads are independent: issue them together (the grid has the table's
  // capacity, so gc is in bounds even past the end of this batch's chunks)
  const int plan_valid = plan.info[1], plan_chunks = plan.info[0];
  const ChunkInfo ci = plan.chunks[gc];
  if (plan_valid == 0 || gc >= plan_chunks) return;
  const int HV = P.HV;
  const int kh = h / (HV / P.HK);
  const int n = ci.n;
  const int64_t t0 = ci.t0;
  constexpr bool delta = DELTA;
  unsigned char* rec = records + (static_cast<int64_t>(gc) * HV + h) * static_cast<int64_t>(REC_BYTES);

  float* sGs = reinterpret_cast<float*>(smem + M::SMALL + O_GS);
  float* sBeta = reinterpret_cast<float*>(smem + M::SMALL + O_BETA);
  float* sRK = reinterpret_cast<float*>(smem + M::SMALL + O_RK);
  float* sRQ = reinterpret_cast<float*>(smem + M::SMALL + O_RQ);
  float* sEG = reinterpret_cast<float*>(smem + M::SMALL + O_EG);
  float* sEGL = reinterpret_cast<float*>(smem + M::SMALL + O_EGL);
  float* sGam = reinterpret_cast<float*>(smem + M::SMALL + O_GAM);
  float* sGA = reinterpret_cast<float*>(smem + M::SMALL + O_GA);
  float* sEA = reinterpret_cast<float*>(smem + M::SMALL + O_EA);
  float* sKF = reinterpret_cast<float*>(smem + M::SMALL + O_KF);
  float* sEL = reinterpret_cast<float*>(smem + M::SMALL + O_EL);
  float* sA = reinterpret_cast<float*>(smem + M::R2);
  float* sT = reinterpret_cast<float*>(smem + M::R2 + SOL_TILE);
  float* sX = reinterpret_cast<float*>(smem + M::R2 + 2 * SOL_TILE);
  constexpr uint32_t KEA = M::KEA;              // K_end (MN-major)
  constexpr uint32_t M_RAW = PERCH ? FrontMap<true>::RAW : 0u;     // raw k | q (per-channel)
  constexpr uint32_t M_SG = PERCH ? FrontMap<true>::S_G : 0u;      // staged log-decay
  constexpr uint32_t M_AK = PERCH ? 0u : FrontMap<false>::AK;      // raw k | q (scalar)
  const int64_t bt = (static_cast<int64_t>(gc) * HV + h) * static_cast<int64_t>(REC_BYTES);
  uint4* blob = reinterpret_cast<uint4*>(records + bt + REC_BLOB) + tid;  // piece p at [p * NT]

  front_issue_loads<PERCH>(P, smem, t0, n, kh, h, tid);
  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, F_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&s_bar, 1);
    tc::mbar_init(&s_bar2, 1);
    tc::mbar_init(&s_ld, 1);
    tc::fence_mbar_init();
    s_abort = 0;
    s_range = 0;
    {                                           // k and q: both 64-channel halves, 64 rows each
      const uint32_t sb = tc::smem_u32(smem + (PERCH ? M_RAW : M_AK));
      const int32_t row0 = static_cast<int32_t>(t0);
      tc::mbar_arrive_expect_tx(&s_ld, 2 * M::AK_HALF + (PERCH ? C * D * 4 : 0));
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        tc::tma_load_3d(sb + a * M::AK_HALF, &tmk, 64 * a, kh, row0, &s_ld);
        tc::tma_load_3d(sb + a * M::AK_HALF + C * 128, &tmq, 64 * a, kh, row0, &s_ld);
      }
      if constexpr (PERCH) {                    // log-decay: four 32-channel quarters
        const uint32_t sg = tc::smem_u32(smem + M_SG);
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) tc::tma_load_3d(sg + qq * (C * 128), &tmg, 32 * qq, h, row0, &s_ld);
      }
    }
  }
  const int row = 32 * (warp & 3) + lane;       // TMEM lane = M row
  const int chalf = warp >> 2;
  const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  uint32_t phase = 0, phase2 = 0;
  auto mma_wait = [&]() {
    const bool ok = tc::mbar_wait_bounded(&s_bar, phase & 1, kWaitLimit);
    phase ^= 1;
    if (!ok) s_abort = 1;
    tc::fence_after_sync();
  };
  auto mma_wait2 = [&]() {                      // the second issuer's group as well
    const bool ok = tc::mbar_wait_bounded(&s_bar, phase & 1, kWaitLimit) &&
                    tc::mbar_wait_bounded(&s_bar2, phase2 & 1, kWaitLimit);
    phase ^= 1;
    phase2 ^= 1;
    if (!ok) s_abort = 1;
    tc::fence_after_sync();
  };
  // 8 raw bf16 channels [c, c + 8) of token i of k or q
  auto kq_off = [&](bool is_q, int i, int c) -> uint32_t {
    return (PERCH ? M_RAW : M_AK) + (c >> 6) * M::AK_HALF + tc::sw128_offset(is_q ? C + i : i, (c & 63) >> 3);
  };
  auto kq_piece = [&](bool is_q, int i, int c) -> const unsigned char* { return smem + kq_off(is_q, i, c); };

  tc::cp_async_wait_all();
  if (!tc::mbar_wait_bounded(&s_ld, 0, kWaitLimit)) s_abort = 1;
  // rows past the chunk's end hold the next sequence's tokens (or the TMA's zero fill):
  // clear them, as a zero-filling copy would, so nothing of another sequence enters
  if (n < C) {
    uint4* ak = reinterpret_cast<uint4*>(smem + (PERCH ? M_RAW : M_AK));
    for (int u = tid; u < (C - n) * 32; u += NT) {        // 2 halves x (k, q) x 8 chunks
      const int r = n + (u >> 5), part = u & 31;
      const int a = part >> 4, qk = (part >> 3) & 1, c8 = part & 7;
      ak[(a * M::AK_HALF + (qk * C + r) * 128) / 16 + c8] = make_uint4(0u, 0u, 0u, 0u);
    }
    if constexpr (PERCH) {                      // log-decay rows: 4 quarters x 8 chunks
      uint4* sgq = reinterpret_cast<uint4*>(smem + M_SG);
      for (int u = tid; u < (C - n) * 32; u += NT) {
        const int r = n + (u >> 5), qq = (u >> 3) & 3, c8 = u & 7;
        sgq[(qq * (C * 128) + r * 128) / 16 + c8] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  __syncthreads();

  // ------------------------------------------------------------------ prep
  {                                             // L2 norms: 4 threads per row
    // lanes l, l + 8, l + 16, l + 24 share row 8 warp + l: each 8-lane group of a 16-byte
    // access reads 8 different rows, whose swizzled chunks fall on different banks
    const int i = 8 * warp + (lane & 7), part = lane >> 3;
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {
      float kx[8], qx[8];
      tc::bf16x8_load(kq_piece(false, i, part * 32 + g8 * 8), kx);
      tc::bf16x8_load(kq_piece(true, i, part * 32 + g8 * 8), qx);
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
  if constexpr (PERCH) {
    float* sG = reinterpret_cast<float*>(smem + M::S_G);
    if (tid < D) {
      // channel tid: inclusive cumsum G, then exp(G - G_a) in place (anchor G_a at the
      // chunk's middle token); exp(G_a) and exp(G_last) go to the small arrays
      float acc = 0.f, gmin = 0.f, gmax = -3.0e38f;
#pragma unroll
      for (int i0 = 0; i0 < C; i0 += 16) {
        float gv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) gv[e] = sG[g_off(i0 + e, tid)];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          acc += gv[e];
          gmin = fminf(gmin, acc);
          gmax = fmaxf(gmax, acc);
          sG[g_off(i0 + e, tid)] = acc;
        }
      }
      const float ga = sG[g_off((n - 1) / 2, tid)];
      if (fmaxf(gmax - ga, ga - gmin) > kMaxHalfChunkDecay) s_range = 1;
#pragma unroll
      for (int i0 = 0; i0 < C; i0 += 16) {
        float gv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) gv[e] = sG[g_off(i0 + e, tid)];
#pragma unroll
        for (int e = 0; e < 16; ++e) sG[g_off(i0 + e, tid)] = __expf(gv[e] - ga);
      }
      sGam[tid] = __expf(acc);
      sGA[tid] = __expf(ga);
      sEL[tid] = __expf(acc - ga);              // exp(G_last - G_a)
    }
  } else if (warp == 0) {                       // scalar: warp scan of 64 values
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
    // anchored factors exp(G_i - G_a), exp(G_a - G_j), anchor mid-chunk, so that
    // exp(G_i - G_j) is a product of two per-token values while both stay finite
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
  if constexpr (PERCH) {
    const float* sG = reinterpret_cast<const float*>(smem + M::S_G);
    {                                           // K- (both halves) first: it reads the raw k rows
      const int j = 8 * warp + (lane & 7), qq = lane >> 3;   // 4 threads per key row
      const float rs = sRK[j];
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        const int cc = 32 * qq + 8 * g8;
        float x[8];
        tc::bf16x8_load(kq_piece(false, j, cc), x);
        const float4 g0 = *reinterpret_cast<const float4*>(sG + g_off(j, cc));
        const float4 g1 = *reinterpret_cast<const float4*>(sG + g_off(j, cc + 4));
        const float f[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float v0 = x[e] * rs * __fdividef(1.f, f[e]);
          const float v1 = x[e + 1] * rs * __fdividef(1.f, f[e + 1]);
          hi[e / 2] = tc::pack_bf16x2(v0, v1);
          const float h0 = __uint_as_float(hi[e / 2] << 16);
          const float h1 = __uint_as_float(hi[e / 2] & 0xffff0000u);
          lo[e / 2] = tc::pack_bf16x2(v0 - h0, v1 - h1);
        }
        *reinterpret_cast<uint4*>(smem + M::BK + tc::cm_offset(j, cc, 128, tc::dense_sbo(D))) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(smem + M::BKLO + tc::cm_offset(j, cc, 128, tc::dense_sbo(D))) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    __syncthreads();
    {                                           // [K+; Q+]: high halves over the raw rows, low to TMEM
      const int i = row < C ? row : row - C;
      const float rs = row < C ? sRK[i] : sRQ[i];
      uint32_t lo[32];
#pragma unroll
      for (int g8 = 0; g8 < 8; ++g8) {
        const int cc = 64 * chalf + 8 * g8;
        unsigned char* piece = const_cast<unsigned char*>(kq_piece(row >= C, i, cc));
        float x[8];
        tc::bf16x8_load(piece, x);
        const float4 g0 = *reinterpret_cast<const float4*>(sG + g_off(i, cc));
        const float4 g1 = *reinterpret_cast<const float4*>(sG + g_off(i, cc + 4));
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
        *reinterpret_cast<uint4*>(piece) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      }
      uint32_t l0[16], l1[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        l0[e] = lo[e];
        l1[e] = lo[16 + e];
      }
      tc::tmem_st16(tmem + lane_addr + F_ALO + 32 * chalf, l0);
      tc::tmem_st16(tmem + lane_addr + F_ALO + 32 * chalf + 16, l1);
      tc::tmem_wait_st();
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // ------------------------------------------------------------------ A-GEMM
  // two issuing threads (one issues a tcgen05.mma only about every 100 cycles), the second
  // into the X columns, which are free until A has been extracted
  if (tid == 0 || tid == 32) {
    const bool second = tid == 32;
    const uint32_t id = tc::idesc_f16(128, 64, tc::kBF16);
    const uint32_t d = tmem + (second ? F_X : F_A);
    if constexpr (PERCH) {
      // [K+; Q+] high halves: the swizzled rows of the raw tiles, K steps of 32 bytes within
      // a 64-channel half
      const uint32_t araw = tc::smem_u32(smem + M::RAW);
      auto dak = [&](int s) {
        return tc::desc_add(tc::smem_desc_sw128(araw + (s >> 2) * M::AK_HALF, 1024), (s & 3) * 32);
      };
      const uint64_t dbk = tc::smem_desc(tc::smem_u32(smem + M::BK), 128, tc::dense_sbo(D));
      const uint64_t dbl = tc::smem_desc(tc::smem_u32(smem + M::BKLO), 128, tc::dense_sbo(D));
      if (!second) {
#pragma unroll
        for (int s = 0; s < D / 16; ++s)        // hi x hi
          tc::mma_ss(d, dak(s), tc::desc_add(dbk, s * 256), id, s > 0);
#pragma unroll
        for (int s = 0; s < D / 32; ++s)        // hi x lo, first half of K
          tc::mma_ss(d, dak(s), tc::desc_add(dbl, s * 256), id, 1);
      } else {
#pragma unroll
        for (int s = D / 32; s < D / 16; ++s)   // hi x lo, second half of K
          tc::mma_ss(d, dak(s), tc::desc_add(dbl, s * 256), id, s > D / 32);
#pragma unroll
        for (int s = 0; s < D / 16; ++s)        // lo x hi (low half from TMEM)
          tc::mma_ts(d, tmem + F_ALO + s * 8, tc::desc_add(dbk, s * 256), id, 1);
      }
    } else {                                    // [K; Q] K^T on the raw rows, one channel half each
      const uint64_t dak = tc::smem_desc_sw128(tc::smem_u32(smem + M::AK) + (second ? M::AK_HALF : 0u), 1024);
#pragma unroll
      for (int s = 0; s < D / 32; ++s)
        tc::mma_ss(d, tc::desc_add(dak, s * 32), tc::desc_add(dak, s * 32), id, s > 0);
    }
    tc::mma_commit(second ? &s_bar2 : &s_bar);
  }
  mma_wait2();

  if constexpr (PERCH) {
    // ---------------------------------------------------------------- K~, Q~, K_end
    // rebuilt from the split halves the A-GEMM has consumed: K~ = K+ exp(G_a) and
    // Q~ = Q+ exp(G_a) (fp16, to the record's [K~; Q~]) and K_end = K- exp(G_last - G_a)
    // (MN-major fp16, over the consumed log-decay)
    {
      const int i = row < C ? row : row - C;
      uint32_t l0[16], l1[16];
      tc::tmem_ld16(tmem + lane_addr + F_ALO + 32 * chalf, l0);
      tc::tmem_ld16(tmem + lane_addr + F_ALO + 32 * chalf + 16, l1);
      tc::tmem_wait_ld();
#pragma unroll
      for (int g8 = 0; g8 < 8; ++g8) {
        const int cc = 64 * chalf + 8 * g8;
        const uint32_t off = kq_off(row >= C, i, cc);
        float x[8];
        tc::bf16x8_load(smem + off, x);
        const float4 a0 = *reinterpret_cast<const float4*>(sGA + cc);
        const float4 a1 = *reinterpret_cast<const float4*>(sGA + cc + 4);
        const float ea[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const uint32_t w = g8 < 4 ? l0[4 * g8 + e / 2] : l1[4 * (g8 - 4) + e / 2];
          x[e] = (x[e] + __uint_as_float(w << 16)) * ea[e];
          x[e + 1] = (x[e + 1] + __uint_as_float(w & 0xffff0000u)) * ea[e + 1];
        }
        if (row < C && !delta) {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
        tc::f16x8_store(rec, REC_KQ + tc::cm_offset(row, cc, 128, KQ_SBO), x);
      }
    }
    {
      const int j = 8 * warp + (lane & 7), qq = lane >> 3;   // 4 threads per key row
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        const int cc = 32 * qq + 8 * g8;
        float hi[8], lo[8], ke[8];
        tc::bf16x8_load(smem + M::BK + tc::cm_offset(j, cc, 128, tc::dense_sbo(D)), hi);
        tc::bf16x8_load(smem + M::BKLO + tc::cm_offset(j, cc, 128, tc::dense_sbo(D)), lo);
        const float4 e0 = *reinterpret_cast<const float4*>(sEL + cc);
        const float4 e1 = *reinterpret_cast<const float4*>(sEL + cc + 4);
        const float el[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) ke[e] = (hi[e] + lo[e]) * el[e];
        tc::f16x8_store(smem, KEA + tc::mn_offset(j, cc, KE_LBO, KE_SBO), ke);
      }
    }
    __syncthreads();                            // the solve tiles and A_qk overwrite K-, k rows
  }

  // ------------------------------------------------------------------ A_kk, A_qk
  {
    uint32_t r0[16], r1[16], q0[16], q1[16];
    tc::tmem_ld16(tmem + lane_addr + F_A + 32 * chalf, r0);
    tc::tmem_ld16(tmem + lane_addr + F_A + 32 * chalf + 16, r1);
    tc::tmem_ld16(tmem + lane_addr + F_X + 32 * chalf, q0);
    tc::tmem_ld16(tmem + lane_addr + F_X + 32 * chalf + 16, q1);
    tc::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      r0[e] = __float_as_uint(__uint_as_float(r0[e]) + __uint_as_float(q0[e]));
      r1[e] = __float_as_uint(__uint_as_float(r1[e]) + __uint_as_float(q1[e]));
    }
    const bool is_k = row < C;
    const int i = is_k ? row : row - C;
    const float ri = is_k ? (PERCH ? 1.f : sRK[i]) * sBeta[i] : (PERCH ? 1.f : sRQ[i]);
    float x[32];
    if (PERCH) {
#pragma unroll
      for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]) * ri;
    } else if (s_anchored) {                    // exp(G_i - G_j) = E_i F_j
      const float rie = ri * sEA[i];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 kf = *reinterpret_cast<const float4*>(sKF + 32 * chalf + e);
        x[e] = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]) * rie * kf.x;
        x[e + 1] = __uint_as_float(e + 1 < 16 ? r0[e + 1] : r1[e - 15]) * rie * kf.y;
        x[e + 2] = __uint_as_float(e + 2 < 16 ? r0[e + 2] : r1[e - 14]) * rie * kf.z;
        x[e + 3] = __uint_as_float(e + 3 < 16 ? r0[e + 3] : r1[e - 13]) * rie * kf.w;
      }
    } else {                                    // exact per pair for extreme decays
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
        *reinterpret_cast<float4*>(sA + sidx(i, 32 * chalf + e)) =
            make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
    } else {
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        tc::f16x8_store(smem, M::LMAT + tc::cm_offset(row, 32 * chalf + 8 * g8, 128, tc::dense_sbo(64)),
                        x + 8 * g8);
    }
  }
  // the 32x32 merge reads the strictly-upper 16x16 blocks of T11 and T22: zero them
  for (int idx = tid; idx < 2 * 256; idx += NT) {
    const int blk = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
    sT[sidx(32 * blk + r, 32 * blk + 16 + c)] = 0.f;
  }
  __syncthreads();

  // ------------------------------------------------------------------ solve
  if (warp < 2) {                               // diagonal 16x16 blocks, one column per lane
    const int base = (warp * 2 + (lane >> 4)) * 16, col = lane & 15;
    // row base + r keeps its columns [base, base + 16) in the 16-float block at base, or at
    // base ^ 16 when r % 8 >= 4, permuted inside it by (r % 4) * 4: constant offsets from
    // two row pointers
    const float* blk0 = sA + base * 64 + base;
    const float* blk1 = sA + base * 64 + (base ^ 16);
    float t[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float* rp = ((r & 4) ? blk1 : blk0) + r * 64;
      float v = r == col ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < r; ++m) v -= rp[m ^ ((r & 3) << 2)] * t[m];
      t[r] = v;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) sT[sidx(base + r, base + col)] = t[r];
  }
  __syncthreads();
  if (tid < 128) {                              // X = A21 T11, two 16x16 pairs
    const int p = tid >> 6, r = (tid >> 2) & 15, c = (tid & 3) * 4;
    const int r0 = 32 * p + 16, c0 = 32 * p;
    float a[16];
#pragma unroll
    for (int m = 0; m < 16; m += 4) {
      const float4 v = *reinterpret_cast<const float4*>(sA + sidx(r0 + r, c0 + m));
      a[m] = v.x; a[m + 1] = v.y; a[m + 2] = v.z; a[m + 3] = v.w;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float4 t = *reinterpret_cast<const float4*>(sT + sidx(c0 + m, c0 + c));
      acc.x += a[m] * t.x; acc.y += a[m] * t.y; acc.z += a[m] * t.z; acc.w += a[m] * t.w;
    }
    *reinterpret_cast<float4*>(sX + (16 * p + r) * XP + c) = acc;
  }
  __syncthreads();
  if (tid < 128) {                              // T21 = -T22 X
    const int p = tid >> 6, r = (tid >> 2) & 15, c = (tid & 3) * 4;
    const int r0 = 32 * p + 16, c0 = 32 * p;
    float a[16];
#pragma unroll
    for (int m = 0; m < 16; m += 4) {
      const float4 v = *reinterpret_cast<const float4*>(sT + sidx(r0 + r, r0 + m));
      a[m] = v.x; a[m + 1] = v.y; a[m + 2] = v.z; a[m + 3] = v.w;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float4 x = *reinterpret_cast<const float4*>(sX + (16 * p + m) * XP + c);
      acc.x += a[m] * x.x; acc.y += a[m] * x.y; acc.z += a[m] * x.z; acc.w += a[m] * x.w;
    }
    *reinterpret_cast<float4*>(sT + sidx(r0 + r, c0 + c)) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
  __syncthreads();
  {                                             // X = A21 T11, one 32x32 pair
    const int r = tid >> 3, c = (tid & 7) * 4;
    float a[32];
#pragma unroll
    for (int m = 0; m < 32; m += 4) {
      const float4 v = *reinterpret_cast<const float4*>(sA + sidx(32 + r, m));
      a[m] = v.x; a[m + 1] = v.y; a[m + 2] = v.z; a[m + 3] = v.w;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      const float4 t = *reinterpret_cast<const float4*>(sT + sidx(m, c));
      acc.x += a[m] * t.x; acc.y += a[m] * t.y; acc.z += a[m] * t.z; acc.w += a[m] * t.w;
    }
    *reinterpret_cast<float4*>(sX + r * XP + c) = acc;
  }
  __syncthreads();
  {                                             // T21 = -T22 X
    const int r = tid >> 3, c = (tid & 7) * 4;
    float a[32];
#pragma unroll
    for (int m = 0; m < 32; m += 4) {
      const float4 v = *reinterpret_cast<const float4*>(sT + sidx(32 + r, 32 + m));
      a[m] = v.x; a[m + 1] = v.y; a[m + 2] = v.z; a[m + 3] = v.w;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      const float4 x = *reinterpret_cast<const float4*>(sX + m * XP + c);
      acc.x += a[m] * x.x; acc.y += a[m] * x.y; acc.z += a[m] * x.z; acc.w += a[m] * x.w;
    }
    *reinterpret_cast<float4*>(sT + sidx(32 + r, c)) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
  __syncthreads();
  for (int u = tid; u < C * (C / 8); u += NT) { // TB[m][j] = T[m][j] beta_j, row pieces
    const int m = (u >> 6) * 8 + (u & 7), j0 = ((u >> 3) & 7) * 8;
    const float4 t0 = *reinterpret_cast<const float4*>(sT + sidx(m, j0));
    const float4 t1 = *reinterpret_cast<const float4*>(sT + sidx(m, j0 + 4));
    const float4 b0 = *reinterpret_cast<const float4*>(sBeta + j0);
    const float4 b1 = *reinterpret_cast<const float4*>(sBeta + j0 + 4);
    const float tv[8] = {t0.x * b0.x, t0.y * b0.y, t0.z * b0.z, t0.w * b0.w,
                         t1.x * b1.x, t1.y * b1.y, t1.z * b1.z, t1.w * b1.w};
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = j0 + e <= m ? tv[e] : 0.f;   // T is lower triangular
    tc::f16x8_store(smem, M::TBT + tc::mn_offset(m, j0, TB_LBO, TB_SBO), x);
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // ------------------------------------------------------------------ A1o = A_qk TB, Kb = K_end^T TB
  // With W = TB K~ never formed (the chain kernel forms V - K~ S instead), the remaining
  // products are Kb = K_end^T TB and A1o = A_qk TB.  A1o is rows 64-127 of the [*; A_qk] TB
  // product (rows 0-63 of that operand are never read back).
  if (tid == 32) {
    const uint32_t id = tc::idesc_f16(128, 64, tc::kF16, false, false, true);
    const uint64_t dl = tc::smem_desc(tc::smem_u32(smem + M::LMAT), 128, tc::dense_sbo(64));
    const uint64_t dt = tc::smem_desc(tc::smem_u32(smem + M::TBT), TB_LBO, TB_SBO);
#pragma unroll
    for (int s = 0; s < C / 16; ++s)
      tc::mma_ss(tmem + F_X, tc::desc_add(dl, s * 256), tc::desc_add(dt, s * 2 * TB_LBO), id, s > 0);
    tc::mma_commit(&s_bar2);
  }
  // K_end = k^ exp(G_last - G_m): A operand K_end^T, MN-major, into the consumed solve area,
  // row pieces of 8 channels (the per-channel path built it before the A extraction)
  if constexpr (!PERCH) {
    for (int u = tid; u < C * (D / 8); u += NT) {
      const int m = (u >> 7) * 8 + (u & 7), c0 = ((u >> 3) & 15) * 8;
      float x[8];
      tc::bf16x8_load(kq_piece(false, m, c0), x);
      const float fe = sRK[m] * sEGL[m];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= fe;
      tc::f16x8_store(smem, KEA + tc::mn_offset(m, c0, KE_LBO, KE_SBO), x);
    }
  }
  if (tid < D) reinterpret_cast<float*>(rec + REC_GAM)[tid] = sGam[tid];
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) {
    const uint32_t id = tc::idesc_f16(128, 64, tc::kF16, false, true, true);
    const uint64_t dke = tc::smem_desc(tc::smem_u32(smem + KEA), KE_LBO, KE_SBO);
    const uint64_t dtb = tc::smem_desc(tc::smem_u32(smem + M::TBT), TB_LBO, TB_SBO);
#pragma unroll
    for (int s = 0; s < C / 16; ++s)
      tc::mma_ss(tmem + F_A, tc::desc_add(dke, s * 2 * KE_LBO), tc::desc_add(dtb, s * 2 * TB_LBO), id, s > 0);
    tc::mma_commit(&s_bar);
  }
  // while they run: K~ = k^ exp(G_m) and Q~ = q scale/|q| exp(G_m) to the record's [K~; Q~]
  // (the per-channel path wrote both before the A extraction)
  if constexpr (!PERCH) {
    for (int u = tid; u < 2 * C * (D / 8); u += NT) {
      const int r = (u >> 7) * 8 + (u & 7), c0 = ((u >> 3) & 15) * 8;   // r: row of [K~; Q~]
      const bool is_q = r >= C;                 // warp-uniform
      const int m = is_q ? r - C : r;
      float x[8];
      tc::bf16x8_load(kq_piece(is_q, m, c0), x);
      const float f = (delta || is_q) ? (is_q ? sRQ[m] : sRK[m]) * sEG[m] : 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= f;
      tc::f16x8_store(rec, REC_KQ + tc::cm_offset(r, c0, 128, KQ_SBO), x);
    }
  }
  mma_wait2();

  // ------------------------------------------------------------------ Kb, A1o out
  // Kb (fp16): record pieces 0-3; A1o (fp16, rows 64-127 of the product): the record's A1O
  {
    uint32_t r0[16], r1[16];
    tc::tmem_ld16(tmem + lane_addr + F_A + 32 * chalf, r0);
    tc::tmem_ld16(tmem + lane_addr + F_A + 32 * chalf + 16, r1);
    tc::tmem_wait_ld();
    float x[32];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      x[e] = __uint_as_float(r0[e]);
      x[e + 16] = __uint_as_float(r1[e]);
    }
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) blob[g8 * NT] = f16x8_pack(x + 8 * g8);
    if (row >= C) {                             // warp-uniform: warps 2, 3, 6, 7
      tc::tmem_ld16(tmem + lane_addr + F_X + 32 * chalf, r0);
      tc::tmem_ld16(tmem + lane_addr + F_X + 32 * chalf + 16, r1);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        x[e] = __uint_as_float(r0[e]);
        x[e + 16] = __uint_as_float(r1[e]);
      }
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        *reinterpret_cast<uint4*>(rec + REC_A1O + tc::cm_offset(row - C, 32 * chalf + 8 * g8, 128, A1O_SBO)) =
            f16x8_pack(x + 8 * g8);
    }
  }

  if (PERCH && s_range && tid == 0) raise_device_error(P.err, KDA_DEVERR_DECAY_RANGE);
  if (s_abort) {                                // the phases that may have timed out
    tc::mbar_wait_bounded(&s_bar, (phase ^ 1) & 1, kWaitLimit);
    tc::mbar_wait_bounded(&s_bar2, (phase2 ^ 1) & 1, kWaitLimit);
    if (tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, F_COLS);
}

// One CTA per (sequence, value head, 64 value columns), warp-specialised into four
// groups that each run their own loop over the sequence's chunks:
//   compute warps 0-7 keep the state slice in registers (thread = key channel, 32 value
//     columns) and run the sequential part: X = [K~; Q~] S, then E' = V - X[0:64] (warps
//     0, 1, 4, 5, whose TMEM lanes are the chunk's tokens), D = Kb E', S <- diag(gam) S + D,
//     publishing the fp16 copy of S.  Each MMA group is split between threads 0 and 128
//     into separate accumulators (one thread issues a tcgen05.mma only about every 90
//     cycles, slower than the tensor core completes these N = 64 shapes);
//   operand warps 8-11 prepare chunks ahead: values (bf16 -> fp16, fetched two chunks
//     ahead), Kb global -> registers -> tensor memory, gamma -> shared memory;
//   lane 0 of warp 12 bulk-copies [K~; Q~ | A1o] and issues the output MMA: A1o E'
//     accumulates onto rows 64-127 of X, which hold Q~ S, beside the state MMA;
//   output warps 14-15 (TMEM lanes 64-127) move the o rows to global memory.
// The groups hand over through monotonic step counters in shared memory.  Every wait is
// bounded; a timeout sets s_abort, each group leaves its loop at a barrier whose
// reduction makes all of its threads agree (or, for the single issuing thread, at once),
// and the device error word is raised.
template <bool SBF16>
__global__ void __launch_bounds__(tcs::NTC, 1)
    tc_chain_kernel(Problem P, PlanView plan, const unsigned char* records) {
  using namespace tcs;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t s_bar_x;                  // [K~; Q~] S of a chunk: both halves (threads 0, 128)
  __shared__ uint64_t s_bar_s;                  // Kb E' of a chunk: both halves
  __shared__ uint64_t s_bar_o;                  // output MMA of a chunk
  __shared__ uint64_t s_kqa_bar[KQA_SLOTS];     // bulk copies of [K~; Q~ | A1o]
  __shared__ uint64_t s_drain;                  // abort only: every MMA issued so far
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_ready;                       // chunks whose V, Kb and gamma are in place
  __shared__ int s_e_ready;                     // chunks whose E' is in place
  __shared__ int s_ps_done;                     // chunks whose state MMA has completed
  __shared__ int s_o_done;                      // chunks whose output MMA has completed
  __shared__ int s_o_free;                      // chunks whose o rows have left tensor memory

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (plan.info[1] == 0) return;
  const int b = blockIdx.x, h = blockIdx.y, vt = blockIdx.z;
  const int HV = P.HV;
  const uint32_t bos = P.offsets[b], eos = P.offsets[b + 1];
  if (eos <= bos) return;
  const uint32_t nchunks = (eos - bos + C - 1) / C;
  const int64_t c0 = plan.seq_chunk0[b];
  const int64_t sbase = (static_cast<int64_t>(P.slot_idx[b]) * HV + h) * D * D + vt * BV;
  const uint32_t sb = tc::smem_u32(smem);
  float* s_gam = reinterpret_cast<float*>(smem + CH_GAM);
  auto rec = [&](uint32_t c) -> const unsigned char* {
    return records + ((c0 + c) * HV + h) * static_cast<int64_t>(REC_BYTES);
  };
  auto v_off = [](uint32_t c) -> uint32_t { return CH_V + (c % V_SLOTS) * V_BYTES; };
  auto kqa_off = [](uint32_t c) -> uint32_t { return CH_KQA + (c % KQA_SLOTS) * KQA_BYTES; };
  auto chunk_n = [&](uint32_t c) -> int {
    const int64_t t0 = static_cast<int64_t>(bos) + static_cast<int64_t>(c) * C;
    return static_cast<int>(min(static_cast<int64_t>(C), static_cast<int64_t>(eos) - t0));
  };
  auto aborted = [&]() -> bool { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };
  auto wait_flag = [&](int* flag, int target) -> bool {   // bounded
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
      if (*reinterpret_cast<volatile int*>(flag) >= target) {
        __threadfence_block();
        return true;
      }
      if (aborted()) return false;
      __nanosleep(20);
    }
    s_abort = 1;
    return false;
  };
  auto set_flag = [&](int* flag, int value) {
    __threadfence_block();
    *reinterpret_cast<volatile int*>(flag) = value;
  };
  auto wait_bar = [&](uint64_t* bar, uint32_t parity) -> bool {   // bounded
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
      if (tc::mbar_try_wait(bar, parity)) {
        tc::fence_after_sync();
        return true;
      }
      if ((i & 255) == 255 && aborted()) return false;
    }
    s_abort = 1;
    return false;
  };

  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, CH_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&s_bar_x, 2);
    tc::mbar_init(&s_bar_s, 2);
    tc::mbar_init(&s_bar_o, 1);
    for (uint32_t i = 0; i < KQA_SLOTS; ++i) tc::mbar_init(&s_kqa_bar[i], 1);
    tc::mbar_init(&s_drain, 3);
    tc::fence_mbar_init();
    s_abort = 0;
    s_ready = 0;
    s_e_ready = 0;
    s_ps_done = 0;
    s_o_done = 0;
    s_o_free = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  const uint32_t id_s = tc::idesc_f16(128, BV, tc::kF16, false, false, true);   // A in TMEM
  const uint32_t id_k = tc::idesc_f16(128, BV, tc::kF16, false, false, true);   // A K-major smem
  const uint64_t dV0 = tc::smem_desc(sb + CH_V, OP_LBO, OP_SBO);
  const uint64_t dS = tc::smem_desc(sb + CH_ST, OP_LBO, OP_SBO);
  const uint64_t dKQ0 = tc::smem_desc(sb + CH_KQA, 128, KQ_SBO);
  const uint64_t dA10 = tc::smem_desc(sb + CH_KQA + KQ_BYTES - A1O_BYTES, 128, A1O_SBO);
  constexpr int W_OPER = NT / 32, W_ISSUE = W_OPER + NTD / 32, W_OUT = W_ISSUE + 2;

  if (warp >= W_OPER && warp < W_ISSUE) {
    // ------------------------------------------------------------------ operand warps
    const int dt = tid - NT;                    // 0..127
    auto issue_v = [&](uint32_t c) {            // raw bf16 v -> MN-major positions of V[c % 5]
      const int64_t t0 = static_cast<int64_t>(bos) + static_cast<int64_t>(c) * C;
      const int n = chunk_n(c);
      const uint32_t dst = sb + v_off(c);
      for (int u = dt; u < C * (BV / 8); u += NTD) {
        const int m = (u >> 6) * 8 + (u & 7), j0 = ((u >> 3) & 7) * 8;
        const bool live = m < n;
        const int64_t t = live ? t0 + m : t0;
        tc::cp_async16(dst + tc::mn_offset(m, j0, OP_LBO, OP_SBO),
                       static_cast<const uint16_t*>(P.v) + t * P.v_stride + static_cast<int64_t>(h) * D + vt * BV + j0,
                       live ? 16u : 0u);
      }
      tc::cp_async_commit();
    };
    auto convert_v = [&](uint32_t c) {          // bf16 -> fp16 in place
      uint4* p = reinterpret_cast<uint4*>(smem + v_off(c));
      for (int u = dt; u < static_cast<int>(V_BYTES / 16); u += NTD) {
        float x[8];
        tc::bf16x8_load(reinterpret_cast<const unsigned char*>(p + u), x);
        p[u] = f16x8_pack(x);
      }
    };
    // a thread serves TMEM lane 32 (warp & 3) + lane for both column halves, i.e. the Kb
    // pieces of compute threads dt and dt + 128 (4 pieces each), and key channel dt of gamma
    uint4 ablob[2 * BLOB_PIECES];
    float gam_next = 0.f;
    auto load_blob = [&](uint32_t c) {
      const uint4* src = reinterpret_cast<const uint4*>(rec(c) + REC_BLOB) + dt;
#pragma unroll
      for (int p = 0; p < static_cast<int>(BLOB_PIECES); ++p) {
        ablob[p] = __ldg(src + p * NT);
        ablob[BLOB_PIECES + p] = __ldg(src + p * NT + NTD);
      }
      gam_next = __ldg(reinterpret_cast<const float*>(rec(c) + REC_GAM) + dt);
    };
    auto store_blob = [&](uint32_t c) {
      const uint32_t base = tmem + lane_addr + T_A + (c & 1) * A_COLS;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const uint4* a = ablob + ch * BLOB_PIECES;
        uint32_t w[16];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          w[4 * p] = a[p].x; w[4 * p + 1] = a[p].y; w[4 * p + 2] = a[p].z; w[4 * p + 3] = a[p].w;
        }
        tc::tmem_st16(base + 16 * ch, w);
      }
      tc::tmem_wait_st();
    };
    issue_v(0);
    if (nchunks > 1) issue_v(1);
    load_blob(0);
    for (uint32_t q = 0; q < nchunks; ++q) {
      // V(q + 2) into the slot of V(q - 3) (its state and output MMAs are done), then V(q)
      // in place: groups issued after V(q) are V(q + 1) and V(q + 2) where they exist
      bool bad = q >= 3 && !wait_flag(&s_o_done, static_cast<int>(q) - 2);
      // the tensor-memory buffer of q held chunk q - 2, read by that chunk's state MMA
      bad = bad || (q >= 2 && !wait_flag(&s_ps_done, static_cast<int>(q) - 1));
      if (tc::named_sync_or(2, NTD, bad || aborted())) break;
      if (q + 2 < nchunks) issue_v(q + 2);
      const uint32_t newer = min(nchunks - 1, q + 2) - q;
      if (newer == 0) tc::cp_async_wait_all();
      else if (newer == 1) tc::cp_async_wait_one();
      else asm volatile("cp.async.wait_group 2;" ::: "memory");
      tc::named_sync(2, NTD);
      tc::fence_after_sync();
      convert_v(q);
      store_blob(q);
      s_gam[(q % GAM_SLOTS) * D + dt] = gam_next;
      if (q + 1 < nchunks) load_blob(q + 1);
      tc::fence_async_smem();
      tc::fence_before_sync();
      tc::named_sync(2, NTD);
      if (dt == 0) set_flag(&s_ready, static_cast<int>(q) + 1);
    }
    tc::cp_async_wait_all();
  } else if (warp >= W_OUT) {
    // ------------------------------------------------------------------ output warps
    const int dq = tid - NT - NTD - 64;         // 0..63: token row, TMEM lane 64 + dq
    float* op = reinterpret_cast<float*>(smem + CH_OST) + dq * OS;
    for (uint32_t c = 0; c < nchunks; ++c) {
      const bool bad = !wait_bar(&s_bar_o, c & 1);
      if (tc::named_sync_or(3, NTO, bad || aborted())) break;
      if (dq == 0) set_flag(&s_o_done, static_cast<int>(c) + 1);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {          // 16 columns of both partial sums
        uint32_t r0[16], r1[16];
        tc::tmem_ld16(tmem + lane_addr + x_col(c, 0) + 16 * qq, r0);
        tc::tmem_ld16(tmem + lane_addr + x_col(c, 1) + 16 * qq, r1);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(op + 16 * qq + e) =
              make_float4(__uint_as_float(r0[e]) + __uint_as_float(r1[e]),
                          __uint_as_float(r0[e + 1]) + __uint_as_float(r1[e + 1]),
                          __uint_as_float(r0[e + 2]) + __uint_as_float(r1[e + 2]),
                          __uint_as_float(r0[e + 3]) + __uint_as_float(r1[e + 3]));
      }
      tc::fence_before_sync();
      tc::named_sync(3, NTO);
      if (dq == 0) set_flag(&s_o_free, static_cast<int>(c) + 1);
      // thread dq stores columns 4 (dq % 16) .. + 3 of rows dq / 16 + 4 k: one pointer step
      // per row group, the partial-chunk test hoisted out of the full chunks
      const int64_t t0 = static_cast<int64_t>(bos) + static_cast<int64_t>(c) * C;
      const int n = chunk_n(c);
      const int i0 = dq >> 4, q4 = dq & 15;
      float* gp = P.o + ((t0 + i0) * HV + h) * D + vt * BV + q4 * 4;
      const float* sp = reinterpret_cast<const float*>(smem + CH_OST) + i0 * OS + q4 * 4;
      const int64_t gstep = static_cast<int64_t>(NTO / 16) * HV * D;
      if (n == C) {
#pragma unroll
        for (int k = 0; k < C / (NTO / 16); ++k)
          *reinterpret_cast<float4*>(gp + k * gstep) = *reinterpret_cast<const float4*>(sp + k * (NTO / 16) * OS);
      } else {
        for (int k = 0; i0 + k * (NTO / 16) < n; ++k)
          *reinterpret_cast<float4*>(gp + k * gstep) = *reinterpret_cast<const float4*>(sp + k * (NTO / 16) * OS);
      }
      tc::named_sync(3, NTO);                   // staging reads done before it is refilled
    }
  } else if (warp == W_ISSUE) {
    // ------------------------------------------------------------------ output-MMA issuer
    if (lane == 0) {
      auto load_kqa = [&](uint32_t c) {         // [K~; Q~ | A1o] of chunk c, one bulk copy
        tc::mbar_arrive_expect_tx(&s_kqa_bar[c % KQA_SLOTS], KQA_BYTES);
        tc::bulk_load(sb + kqa_off(c), rec(c) + REC_KQ, KQA_BYTES, &s_kqa_bar[c % KQA_SLOTS]);
      };
      for (uint32_t q = 0; q < min(nchunks, KQA_SLOTS); ++q) load_kqa(q);
      for (uint32_t c = 0; c < nchunks; ++c) {
        // the slot of chunk c - 1 takes chunk c + 2 as soon as that chunk's output MMA is done
        // (about when chunk c starts): two chunk periods ahead of its use
        if (c >= 1 && c + 2 < nchunks) {
          if (!wait_flag(&s_o_done, static_cast<int>(c))) break;
          load_kqa(c + 2);
        }
        // E'(c) in place (so X(c) is complete and its rows 0-63 consumed); o rows of c - 1
        // out, which keeps the completion barrier one phase ahead of its waiters
        if (!wait_flag(&s_e_ready, static_cast<int>(c) + 1)) break;
        if (!wait_flag(&s_o_free, static_cast<int>(c))) break;
        if (!wait_bar(&s_kqa_bar[c % KQA_SLOTS], (c / KQA_SLOTS) & 1)) break;
        const uint64_t da = tc::desc_add(dA10, (c % KQA_SLOTS) * KQA_BYTES);
        const uint64_t dv = tc::desc_add(dV0, (c % V_SLOTS) * V_BYTES);
#pragma unroll
        for (int s = 0; s < C / 16; ++s)
          tc::mma_ss(tmem + x_col(c, 0), tc::desc_add(da, s * 256), tc::desc_add(dv, s * 2 * OP_LBO), id_k, 1);
        tc::mma_commit(&s_bar_o);
      }
    }
  } else if (warp < W_OPER) {
    // ------------------------------------------------------------------ compute warps
    const int row = 32 * (warp & 3) + lane;     // TMEM lane = key channel (state row)
    const int chalf = warp >> 2;
    const int part = tid >> 7;                  // threads 0 and 128 issue one half each
    const bool extract = row < C;               // warps 0, 1, 4, 5: row = token of X, E'
    float Sv[32];
    {
      const int64_t base = sbase + static_cast<int64_t>(row) * D + 32 * chalf;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        Sv[j] = SBF16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(P.pool)[base + j])
                      : static_cast<const float*>(P.pool)[base + j];
    }
    auto write_state_operand = [&]() {          // S, fp16, MN-major
#pragma unroll
      for (int p = 0; p < 4; ++p)
        *reinterpret_cast<uint4*>(smem + CH_ST + tc::mn_offset(row, 32 * chalf + 8 * p, OP_LBO, OP_SBO)) =
            f16x8_pack(Sv + 8 * p);
    };
    write_state_operand();
    tc::fence_async_smem();
    tc::fence_before_sync();
    tc::named_sync(1, NT);
    tc::fence_after_sync();
    bool stop = false;
    for (uint32_t c = 0; c < nchunks && !stop; ++c) {
      bool bad = false;
      if ((tid & 127) == 0) {                   // X = [K~; Q~] S, K half `part`
        // [K~; Q~ | A1o](c) in place; X(c & 1) free once the o rows of chunk c - 2 are out
        bad = !wait_bar(&s_kqa_bar[c % KQA_SLOTS], (c / KQA_SLOTS) & 1);
        bad = bad || (c >= 2 && !wait_flag(&s_o_free, static_cast<int>(c) - 1));
        if (!bad) {
          tc::fence_after_sync();
          const uint64_t da = tc::desc_add(dKQ0, (c % KQA_SLOTS) * KQA_BYTES);
#pragma unroll
          for (int s = 4 * part; s < 4 * part + 4; ++s)
            tc::mma_ss(tmem + x_col(c, part), tc::desc_add(da, s * 256), tc::desc_add(dS, s * 2 * OP_LBO),
                       id_k, s > 4 * part);
          tc::mma_commit(&s_bar_x);
        }
      }
      if (extract) {                            // E' = V - K~ S over V's slot
        bad = bad || !wait_bar(&s_bar_x, c & 1);
        bad = bad || !wait_flag(&s_ready, static_cast<int>(c) + 1);   // V(c), Kb(c)
        bad = __any_sync(0xffffffffu, bad);     // tcgen05.ld is warp-collective
        if (!bad) {
          unsigned char* vp = smem + v_off(c);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t r0[16], r1[16];
            tc::tmem_ld16(tmem + lane_addr + x_col(c, 0) + 32 * chalf + 16 * hh, r0);
            tc::tmem_ld16(tmem + lane_addr + x_col(c, 1) + 32 * chalf + 16 * hh, r1);
            tc::tmem_wait_ld();
#pragma unroll
            for (int p = 0; p < 2; ++p) {
              const uint32_t off = tc::mn_offset(row, 32 * chalf + 16 * hh + 8 * p, OP_LBO, OP_SBO);
              float v[8];
              tc::f16x8_load(vp + off, v);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                v[e] -= __uint_as_float(r0[8 * p + e]) + __uint_as_float(r1[8 * p + e]);
              *reinterpret_cast<uint4*>(vp + off) = f16x8_pack(v);
            }
          }
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        bad = tc::named_sync_or(4, NT / 2, bad || aborted());
        tc::fence_after_sync();
        if (!bad && (tid & 127) == 0) {         // D = Kb E', K half `part`
          if (tid == 0) set_flag(&s_e_ready, static_cast<int>(c) + 1);
          const uint32_t ta = tmem + T_A + (c & 1) * A_COLS;
          const uint64_t dv = tc::desc_add(dV0, (c % V_SLOTS) * V_BYTES);
#pragma unroll
          for (int s = 2 * part; s < 2 * part + 2; ++s)
            tc::mma_ts(tmem + (part ? T_DS2 : T_DS), ta + s * 8, tc::desc_add(dv, s * 2 * OP_LBO), id_s,
                       s > 2 * part);
          tc::mma_commit(&s_bar_s);
        }
      }
      bad = bad || !wait_bar(&s_bar_s, c & 1);
      bad = bad || !wait_flag(&s_ready, static_cast<int>(c) + 1);     // gamma(c)
      bad = __any_sync(0xffffffffu, bad);
      if (!bad) {
        if (tid == 0) set_flag(&s_ps_done, static_cast<int>(c) + 1);
        uint32_t r0[16], r1[16], q0[16], q1[16];
        tc::tmem_ld16(tmem + lane_addr + T_DS + 32 * chalf, r0);
        tc::tmem_ld16(tmem + lane_addr + T_DS + 32 * chalf + 16, r1);
        tc::tmem_ld16(tmem + lane_addr + T_DS2 + 32 * chalf, q0);
        tc::tmem_ld16(tmem + lane_addr + T_DS2 + 32 * chalf + 16, q1);
        tc::tmem_wait_ld();
        const float gam = s_gam[(c % GAM_SLOTS) * D + row];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          Sv[e] = gam * Sv[e] + (__uint_as_float(r0[e]) + __uint_as_float(q0[e]));
          Sv[e + 16] = gam * Sv[e + 16] + (__uint_as_float(r1[e]) + __uint_as_float(q1[e]));
        }
        // S(c) was read only by X(c), complete before Kb E'(c) was issued
        if (c + 1 < nchunks) write_state_operand();
      }
      tc::fence_async_smem();
      tc::fence_before_sync();
      stop = tc::named_sync_or(1, NT, bad || aborted());
      tc::fence_after_sync();
    }
    if (!aborted()) {
      const int64_t base = sbase + static_cast<int64_t>(row) * D + 32 * chalf;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (SBF16)
          static_cast<uint16_t*>(P.pool)[base + j] = f32_to_bf16_bits(Sv[j]);
        else
          static_cast<float*>(P.pool)[base + j] = Sv[j];
      }
    }
  }

  __syncthreads();
  if (s_abort) {
    // let whatever is still in flight finish (bounded) before shared and tensor memory go:
    // every MMA of the three issuing threads (one commit each on the drain barrier) and the
    // bulk copies (both phases of their barriers)
    if (tid == 0 || tid == 128 || tid == 32 * W_ISSUE) tc::mma_commit(&s_drain);
    tc::mbar_wait_bounded(&s_drain, 0, kWaitLimit);
    for (uint32_t k = 0; k < 2; ++k)
      for (uint32_t i = 0; i < KQA_SLOTS; ++i) tc::mbar_wait_bounded(&s_kqa_bar[i], k, kWaitLimit);
    if (tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, CH_COLS);
}

size_t split_workspace_bytes(const Problem& P) {
  const size_t off = plan_layout(P, nullptr, 0, nullptr);
  return off + static_cast<size_t>(plan_max_chunks(P)) * static_cast<size_t>(P.HV) * tcs::REC_BYTES;
}

// cuTensorMapEncodeTiled from the driver (the runtime is linked statically, libcuda is not)
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [T, HK, 128] bf16 rows with a row stride of `stride` elements: boxes of 64 channels x
// 1 head x 64 tokens, 128-byte swizzle, zero fill past the last token
static bool encode_rows_map(CUtensorMap* m, const void* base, const Problem& P, int64_t stride) {
  auto enc = tensor_map_encoder();
  if (!enc || P.T <= 0) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(tcs::D), static_cast<cuuint64_t>(P.HK),
                              static_cast<cuuint64_t>(P.T)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(tcs::D) * 2, static_cast<cuuint64_t>(stride) * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(tcs::C)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// per-channel log-decay [T, HV, 128] fp32: boxes of 32 channels x 1 head x 64 tokens, 128-byte
// swizzle, zero fill past the last token
static bool encode_g_map(CUtensorMap* m, const Problem& P) {
  auto enc = tensor_map_encoder();
  if (!enc || P.T <= 0) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(tcs::D), static_cast<cuuint64_t>(P.HV),
                              static_cast<cuuint64_t>(P.T)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(tcs::D) * 4,
                                 static_cast<cuuint64_t>(P.HV) * tcs::D * 4};
  const cuuint32_t box[3] = {32, 1, static_cast<cuuint32_t>(tcs::C)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(P.g), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool PERCH, bool DELTA>
static cudaError_t launch_front_t(const Problem& P, const PlanView& plan, unsigned char* recs,
                                  cudaStream_t st) {
  auto k = tc_front_kernel<PERCH, DELTA>;
  constexpr uint32_t bytes = tcs::FrontMap<PERCH>::BYTES + 1024;
  alignas(64) CUtensorMap tmq, tmk, tmg;
  memset(&tmg, 0, sizeof(tmg));
  if (!(encode_rows_map(&tmq, P.q, P, P.q_stride) && encode_rows_map(&tmk, P.k, P, P.k_stride)))
    return cudaErrorInvalidValue;
  if (PERCH && !encode_g_map(&tmg, P)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  k<<<dim3(static_cast<unsigned>(plan_max_chunks(P)), P.HV), tcs::NT, bytes, st>>>(P, plan, recs, tmq, tmk, tmg);
  return cudaGetLastError();
}

template <bool SBF16>
static cudaError_t launch_chain_t(const Problem& P, const PlanView& plan, const unsigned char* recs,
                                  cudaStream_t st) {
  auto k = tc_chain_kernel<SBF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(tcs::CH_BYTES));
  if (e != cudaSuccess) return e;
  k<<<dim3(P.num_seqs, P.HV, tcs::D / tcs::BV), tcs::NTC, tcs::CH_BYTES, st>>>(P, plan, recs);
  return cudaGetLastError();
}

cudaError_t launch_prefill_split(const Problem& P, void* workspace, bool perch, bool sbf16,
                                 cudaStream_t stream, const Stages& st) {
  PlanView plan;
  const size_t off = plan_layout(P, static_cast<char*>(workspace), 0, &plan);
  unsigned char* recs = static_cast<unsigned char*>(workspace) + off;
  st.mark(0, stream);
  cudaError_t e = launch_plan(P, plan, stream);
  if (e != cudaSuccess) return e;
  st.mark(1, stream);
  const bool delta = !(P.flags & KDA_FLAG_NO_DELTA);
  e = perch ? (delta ? launch_front_t<true, true>(P, plan, recs, stream)
                     : launch_front_t<true, false>(P, plan, recs, stream))
            : (delta ? launch_front_t<false, true>(P, plan, recs, stream)
                     : launch_front_t<false, false>(P, plan, recs, stream));
  if (e != cudaSuccess) return e;
  st.mark(2, stream);
  e = sbf16 ? launch_chain_t<true>(P, plan, recs, stream) : launch_chain_t<false>(P, plan, recs, stream);
  st.mark(3, stream);
  return e;
}

}  // namespace kda
