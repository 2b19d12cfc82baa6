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
#include "kda_common.cuh"
#include "prefill_plan.cuh"
#include "tc_utils.cuh"
#include "tma_maps.cuh"

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
constexpr float kMaxHalfChunkDecay = 80.0f;   // scalar decay: anchored factors in fp32

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

// per-chunk vectors of the scalar-decay front kernel (byte offsets inside its SMALL area)
constexpr uint32_t O_GS = 0, O_BETA = 256, O_RK = 512, O_RQ = 768, O_EG = 1024, O_EGL = 1280,
                   O_GAM = 1536, O_EA = 2560, O_KF = 2816, SMALL_BYTES = 3584;

// Per-channel decay: the chunk's 64 tokens form four sub-blocks of 16.  Rows of sub-block I
// carry their decay relative to the last token before it (G_ref(I): 0 for I = 0, else
// G_{16I-1}), so that for a key j of an earlier sub-block J < I
//   exp(G_i - G_j) = exp(G_i - G_ref(I)) * exp(G_ref(I) - G_j),   both factors <= 1,
// and fp16 operands hold them whatever the decay.  Pairs inside one sub-block use the column
// factor exp(G_ref(J) - G_j) >= 1, which fp16 holds as long as a channel decays by at most
// kSubBlockDecay nats from the reference to any token of the sub-block; the (sub-block,
// channel) pairs above it are summed exactly in fp32 instead (exp per pair).  The row
// operand is scaled by 2^8 and the column operands by 2^-8 (the product is unchanged), which
// keeps the small row factors of a strongly decaying channel out of fp16's subnormal range.
constexpr float kSubBlockDecay = 12.0f;
constexpr float kLog2e = 1.4426950408889634f;   // the per-channel path keeps G in log2 units
constexpr float kRowScale = 256.0f, kColScale = 1.0f / 256.0f;
// The factors above are <= 1 only for a non-increasing cumulative log-decay: a per-channel
// log-decay above this bound (a gate above 1) is outside the tensor-core path's domain.
constexpr float kMaxLogDecay = 1.0f / 64.0f;
// per-chunk vectors of the per-channel front kernel (byte offsets inside its SMALL area):
//   BETA, RK, RQ  beta, 1/|k|, scale/|q| per token
//   GB   G at tokens 15, 31 and, relative to token 31, at 47, 63 per channel (the sub-block
//        boundaries; each 32-token half keeps its own cumulative sum)
//   ES   exp(G_15), exp(G_31), exp(G_47) (K~ and Q~ of sub-blocks 1-3 from their row factors)
//   W    diagonal column factor exp(G_ref(J) - G_end(J)) of sub-block J (0 for exact channels)
//   F    exp(G_ref(I) - G_end(J)) for (I, J) = (2, 0), (3, 0), (3, 1) (I = J + 1 needs none)
//   MASK exact channels: 4 words of 32 channels per sub-block
constexpr uint32_t P_BETA = 0, P_RK = 256, P_RQ = 512, P_GB = 768, P_ES = P_GB + 4 * 512,
                   P_W = P_ES + 3 * 512, P_F = P_W + 4 * 512, P_MASK = P_F + 3 * 512,
                   SMALL_PC_BYTES = P_MASK + 4 * 4 * 4;
// the off-diagonal column operand holds the six (I, J) pairs J < I, 16 rows each
__host__ __device__ constexpr int off_slot(int I, int J) { return I * (I - 1) / 2 + J; }

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
  static constexpr uint32_t BETA = SMALL + O_BETA, RK = SMALL + O_RK, RQ = SMALL + O_RQ;
};

// Per-channel decay: TMA copies stage the raw k and q rows (the 128-byte swizzled layout of
// the scalar path) and the log-decay rows (four 32-channel quarters, each 64 rows of 128
// bytes, swizzled the same way).  The log-decay becomes G in place; the row operand R
// (fp16) overwrites the raw rows in place; once every thread holds its G pieces, the
// diagonal column operand goes over G and the off-diagonal one beside it.  After the A-GEMM
// the solve tiles reuse both column operands and TB / [*; A_qk] the rows.  K_end lives in
// tensor memory.
template <>
struct FrontMap<true> {
  static constexpr uint32_t AK_HALF = 128 * 128;
  static constexpr uint32_t RAW = 0;                    // raw k | q -> R; then TB, [*; A_qk]
  static constexpr uint32_t S_G = RAW + 2 * AK_HALF;    // log-decay -> G -> C_diag; then solve
  static constexpr uint32_t CD = S_G;                   // C_diag 64 x 128 fp16, K-major
  static constexpr uint32_t CO = S_G + C * D * 4;       // C_off 96 x 128 fp16, K-major
  static constexpr uint32_t SMALL = CO + 6 * 16 * D * 2;
  static constexpr uint32_t BYTES = SMALL + SMALL_PC_BYTES;
  static constexpr uint32_t R2 = S_G;
  static constexpr uint32_t TBT = RAW;
  static constexpr uint32_t LMAT = RAW + AK_HALF - 64 * 64 * 2;   // rows 64-127: half 1 k rows
  static constexpr uint32_t BETA = SMALL + P_BETA, RK = SMALL + P_RK, RQ = SMALL + P_RQ;
  static_assert(R2 + SOL_BYTES <= SMALL, "solve tiles inside the consumed column operands");
  static_assert(CD + C * D * 2 <= CO, "diagonal column operand inside the consumed G");
};

// front TMEM columns.  Scalar decay: A_kk/A_qk (second issuer's half of K in F_X), then
// Kb | A1o.  Per-channel decay: the diagonal products (F_D, 64 columns: sub-block J at
// 16 J) and the off-diagonal ones (F_O, 96 columns: pair (I, J) at 16 off_slot(I, J)), then
// Kb | A1o over them; K_end^T (lane = channel, 64 tokens as fp16 pairs) at F_KE.
constexpr uint32_t F_A = 0, F_X = 64, F_D = 0, F_O = 64, F_KE = 160, F_COLS = 256;
static_assert(F_O + 96 <= F_KE && F_KE + 32 <= F_COLS, "front tensor-memory columns");

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
    tc::cp_async4(sb + M::BETA + tid * 4, P.beta + t * HV + h, live ? 4u : 0u);
    if (!PERCH) tc::cp_async4(sb + FrontMap<false>::SMALL + O_GS + tid * 4, P.g + t * HV + h, live ? 4u : 0u);
  }
  tc::cp_async_commit();
}

__device__ __forceinline__ void load8(float* x, const float* p) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// One CTA per (chunk, value head): everything of the chunk that does not depend on the
// state, written to the chunk's record.
// DELTA = false is the additive write (no delta rule): A_kk = 0 makes T = I and K~ = 0
// drops W = TB K~; a template parameter, so that the delta rule's code carries no test of it
template <bool PERCH, bool DELTA>
__global__ void __launch_bounds__(tcs::NT, 2)
    tc_front_kernel(Problem P, PlanView plan, unsigned char* records,
                    const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmg, int ahead) {
  using namespace tcs;
  using M = FrontMap<PERCH>;
  using MS = FrontMap<false>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzled operand needs a 1024-byte aligned base; the launch adds 1 KB of slack
  unsigned char* const smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t s_bar;                    // MMAs issued by thread 0
  __shared__ uint64_t s_bar2;                   // MMAs issued by thread 32
  __shared__ uint64_t s_ld;                     // TMA copies of k and q (and g)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_range;                       // per-channel: a log-decay above kMaxLogDecay
  __shared__ int s_anchored;                    // scalar: anchored factors in range
  __shared__ int s_anyslow;                     // per-channel: some pair summed exactly

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

  float* sBeta = reinterpret_cast<float*>(smem + M::BETA);
  float* sRK = reinterpret_cast<float*>(smem + M::RK);
  float* sRQ = reinterpret_cast<float*>(smem + M::RQ);
  float* sA = reinterpret_cast<float*>(smem + M::R2);
  float* sT = reinterpret_cast<float*>(smem + M::R2 + SOL_TILE);
  float* sX = reinterpret_cast<float*>(smem + M::R2 + 2 * SOL_TILE);
  // scalar decay only
  float* sGs = reinterpret_cast<float*>(smem + MS::SMALL + O_GS);
  float* sEG = reinterpret_cast<float*>(smem + MS::SMALL + O_EG);
  float* sEGL = reinterpret_cast<float*>(smem + MS::SMALL + O_EGL);
  float* sGam = reinterpret_cast<float*>(smem + MS::SMALL + O_GAM);
  float* sEA = reinterpret_cast<float*>(smem + MS::SMALL + O_EA);
  float* sKF = reinterpret_cast<float*>(smem + MS::SMALL + O_KF);
  constexpr uint32_t M_RAW = PERCH ? FrontMap<true>::RAW : 0u;     // raw k | q (per-channel)
  constexpr uint32_t M_SG = PERCH ? FrontMap<true>::S_G : 0u;      // staged log-decay
  constexpr uint32_t M_AK = PERCH ? 0u : FrontMap<false>::AK;      // raw k | q (scalar)
  uint4* blob = reinterpret_cast<uint4*>(rec + REC_BLOB) + tid;    // piece p at [p * NT]

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
    s_anyslow = 0;
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
  if (tid == 32 && ahead > 0) {
    // CTAs start in the order of their linear index, `ahead` of them resident at once: the
    // one `ahead` places later starts about when this one ends, so its k, q (and log-decay)
    // tiles go to L2 now and its own copies find them there
    const int64_t L = static_cast<int64_t>(h) * gridDim.x + gc + ahead;
    const int gn = static_cast<int>(L % gridDim.x), hn = static_cast<int>(L / gridDim.x);
    if (hn < HV && gn < plan_chunks) {
      const int32_t rn = static_cast<int32_t>(plan.chunks[gn].t0);
      const int khn = hn / (HV / P.HK);
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        tc::tma_prefetch_3d(&tmk, 64 * a, khn, rn);
        tc::tma_prefetch_3d(&tmq, 64 * a, khn, rn);
      }
      if constexpr (PERCH) {
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) tc::tma_prefetch_3d(&tmg, 32 * qq, hn, rn);
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
  auto mma_wait2 = [&]() {                      // both issuers' groups
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
    float* sGB = reinterpret_cast<float*>(smem + M::SMALL + P_GB);
    float* sES = reinterpret_cast<float*>(smem + M::SMALL + P_ES);
    float* sW = reinterpret_cast<float*>(smem + M::SMALL + P_W);
    float* sF = reinterpret_cast<float*>(smem + M::SMALL + P_F);
    uint32_t* sMask = reinterpret_cast<uint32_t*>(smem + M::SMALL + P_MASK);
    {
      // ---------------------------------------------------------------- cumulative log-decay
      // thread = (channel c, token half hh): each half sums its own 32 tokens.  Every
      // quantity inside a half (the sub-blocks' row and column factors, the exact diagonal
      // pairs) depends only on differences within it, so G stays half-local in shared memory
      // and GB holds, per channel, G_15 and G_31 of the first half and the second half's local
      // G_47 and G_63; the cross-half values below add the first half's total G_31.
      const int c = tid & 127, hh = tid >> 7;
      float gv[32];
      bool rise = false;
#pragma unroll
      for (int e = 0; e < 32; ++e) gv[e] = sG[g_off(32 * hh + e, c)];
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {            // G in log2 units: every factor is one ex2
        rise = rise || gv[e] > kMaxLogDecay;
        acc = fmaf(gv[e], kLog2e, acc);
        gv[e] = acc;
      }
      float m0 = gv[0], m1 = gv[16];            // lowest G of each of the half's sub-blocks
#pragma unroll
      for (int e = 1; e < 16; ++e) {
        m0 = fminf(m0, gv[e]);
        m1 = fminf(m1, gv[16 + e]);
      }
      if (rise) s_range = 1;
#pragma unroll
      for (int e = 0; e < 32; ++e) sG[g_off(32 * hh + e, c)] = gv[e];
      sGB[(2 * hh) * 128 + c] = gv[15];
      sGB[(2 * hh + 1) * 128 + c] = gv[31];
      // sub-blocks 2 hh and 2 hh + 1 (half-local: reference 0 and gv[15], ends gv[15], gv[31]):
      // a channel whose decay from the sub-block's reference to any of its tokens exceeds
      // kSubBlockDecay is summed exactly on the diagonal
      const bool slow0 = -m0 > kSubBlockDecay * kLog2e, slow1 = gv[15] - m1 > kSubBlockDecay * kLog2e;
      const uint32_t b0 = __ballot_sync(0xffffffffu, slow0), b1 = __ballot_sync(0xffffffffu, slow1);
      if (lane == 0) {
        sMask[(2 * hh) * 4 + (warp & 3)] = b0;
        sMask[(2 * hh + 1) * 4 + (warp & 3)] = b1;
        if (b0 | b1) s_anyslow = 1;
      }
      sW[(2 * hh) * 128 + c] = slow0 ? 0.f : ex2(-gv[15]);
      sW[(2 * hh + 1) * 128 + c] = slow1 ? 0.f : ex2(gv[15] - gv[31]);
      __syncthreads();
      const float g15 = sGB[c], g31 = sGB[128 + c], l47 = sGB[256 + c], l63 = sGB[384 + c];
      if (hh == 0) {
        sES[c] = ex2(g15);
        sES[128 + c] = ex2(g31);
        sF[c] = ex2(g31 - g15);                 // sub-block 0 seen from sub-block 2
      } else {
        sES[256 + c] = ex2(g31 + l47);
        sF[128 + c] = ex2(g31 + l47 - g15);     // sub-block 0 seen from sub-block 3
        sF[256 + c] = ex2(l47);                 // sub-block 1 seen from sub-block 3
        reinterpret_cast<float*>(rec + REC_GAM)[c] = ex2(g31 + l63);
      }
      // the chunk's last G in this half's coordinates
      const float g63 = hh == 0 ? g31 + l63 : l63;
      // K_end = k^ exp(G_last - G_j) of this thread's 32 tokens in channel c, to tensor
      // memory (lane = channel c, two tokens per column): the A operand of K_end^T TB
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const int j = 32 * hh + e;
        const float2 rk = *reinterpret_cast<const float2*>(sRK + j);
        const float2 kj = make_float2(tc::bf16_at(smem, kq_off(false, j, c), c & 7),
                                      tc::bf16_at(smem, kq_off(false, j + 1, c), c & 7));
        const float2 x = mul2(mul2(kj, rk), make_float2(ex2(g63 - gv[e]), ex2(g63 - gv[e + 1])));
        w[e / 2] = tc::pack_f16x2(x.x, x.y);
      }
      tc::tmem_st16(tmem + lane_addr + F_KE + 16 * hh, w);
      tc::tmem_wait_st();
    }
    __syncthreads();

    if (s_anyslow) {
      // ---------------------------------------------------------------- exact diagonal pairs
      // thread = (row of [K; Q], 8 keys of its row's sub-block): the channels above the
      // threshold, exp(G_i - G_j) per pair in fp32; the sums initialise the diagonal
      // accumulator (zeros elsewhere), onto which the A-GEMM adds the other channels
      const int jh = warp >> 2, p = (warp & 3) & 1;
      const bool is_q = row >= C;
      const int i = row & (C - 1), I = i >> 4, jb = 16 * I + 8 * jh;
      const float rs = is_q ? sRQ[i] : sRK[i];
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
      for (int w4 = 0; w4 < 4; ++w4) {
        uint32_t bits = sMask[I * 4 + w4];
        while (bits) {
          const int cc = 32 * w4 + __ffs(bits) - 1;
          bits &= bits - 1;
          const float xi = tc::bf16_at(smem, kq_off(is_q, i, cc), cc & 7) * rs;
          const float gi = sG[g_off(i, cc)];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = jb + e;
            if (is_q ? j <= i : j < i)
              acc[e] += xi * tc::bf16_at(smem, kq_off(false, j, cc), cc & 7) * sRK[j] *
                        ex2(gi - sG[g_off(j, cc)]);
          }
        }
      }
      const bool lo = (I & 1) == 0;             // this lane's sub-block is 2p, else 2p + 1
      uint32_t v0[8], v1[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v0[e] = lo ? __float_as_uint(acc[e]) : 0u;
        v1[e] = lo ? 0u : __float_as_uint(acc[e]);
      }
      tc::tmem_st8(tmem + lane_addr + F_D + 32 * p + 8 * jh, v0);
      tc::tmem_st8(tmem + lane_addr + F_D + 32 * p + 16 + 8 * jh, v1);
      tc::tmem_wait_st();
    }

    // ---------------------------------------------------------------- operands
    // thread: token jr (8-lane groups cover 8 rows, so the swizzled accesses spread over the
    // banks) and 8-channel pieces c0 = 8 (lane / 8 + 4 it).  First every G piece to registers,
    // since the diagonal column operand is written over G.
    const int jr = 8 * warp + (lane & 7);
    const int J = jr >> 4;                      // warp-uniform
    float gp[4][8];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int c0 = 8 * ((lane >> 3) + 4 * it);
      const float4 a = *reinterpret_cast<const float4*>(sG + g_off(jr, c0));
      const float4 b = *reinterpret_cast<const float4*>(sG + g_off(jr, c0 + 4));
      gp[it][0] = a.x; gp[it][1] = a.y; gp[it][2] = a.z; gp[it][3] = a.w;
      gp[it][4] = b.x; gp[it][5] = b.y; gp[it][6] = b.z; gp[it][7] = b.w;
    }
    __syncthreads();
    {
      const float rk = sRK[jr], rq = sRQ[jr];
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int c0 = 8 * ((lane >> 3) + 4 * it);
        float kx[8], qx[8], gref[8], gend[8], es[8], wd[8];
        tc::bf16x8_load(kq_piece(false, jr, c0), kx);
        tc::bf16x8_load(kq_piece(true, jr, c0), qx);
        load8(gend, sGB + J * 128 + c0);
        load8(wd, sW + J * 128 + c0);
        if (J == 0 || J == 2) {                  // the half's first sub-block: reference 0
#pragma unroll
          for (int e = 0; e < 8; ++e) gref[e] = 0.f;
        } else {
          load8(gref, sGB + (J - 1) * 128 + c0);
        }
        if (J == 0) {
#pragma unroll
          for (int e = 0; e < 8; ++e) es[e] = 1.f;
        } else {
          load8(es, sES + (J - 1) * 128 + c0);
        }
        const uint32_t mb = (sMask[J * 4 + (c0 >> 5)] >> (c0 & 31)) & 0xffu;
        float rkv[8], rqv[8], kt[8], qt[8], ke[8], cd[8];
        const float2 rk2 = make_float2(rk, rk), rq2 = make_float2(rq, rq);
        const float2 rks = make_float2(rk * kRowScale, rk * kRowScale), rqs = make_float2(rq * kRowScale, rq * kRowScale);
        const float2 rkc = make_float2(rk * kColScale, rk * kColScale);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {                   // two channels at a time
          const float2 r = make_float2(ex2(gp[it][e] - gref[e]), ex2(gp[it][e + 1] - gref[e + 1]));   // <= 1
          const float2 eps = make_float2(ex2(gend[e] - gp[it][e]), ex2(gend[e + 1] - gp[it][e + 1]));  // <= 1
          const float2 kxr = mul2(make_float2(kx[e], kx[e + 1]), r);
          const float2 qxr = mul2(make_float2(qx[e], qx[e + 1]), r);
          const float2 R_k = mul2(kxr, rks), R_q = mul2(qxr, rqs);
          const float2 es2 = make_float2(es[e], es[e + 1]);
          const float2 K_t = mul2(mul2(kxr, rk2), es2);   // K~ = k^ exp(G_j)
          const float2 Q_t = mul2(mul2(qxr, rq2), es2);   // Q~ = q^ exp(G_j)
          const float2 k_e = mul2(mul2(make_float2(kx[e], kx[e + 1]), eps), rkc);
          const float2 c_d = mul2(k_e, make_float2(wd[e], wd[e + 1]));   // k^ exp(G_ref(J) - G_j) / 256
          rkv[e] = R_k.x; rkv[e + 1] = R_k.y;
          rqv[e] = R_q.x; rqv[e + 1] = R_q.y;
          kt[e] = delta ? K_t.x : 0.f; kt[e + 1] = delta ? K_t.y : 0.f;
          qt[e] = Q_t.x; qt[e + 1] = Q_t.y;
          ke[e] = k_e.x; ke[e + 1] = k_e.y;
          cd[e] = ((mb >> e) & 1u) ? 0.f : c_d.x;
          cd[e + 1] = ((mb >> (e + 1)) & 1u) ? 0.f : c_d.y;
        }
        tc::f16x8_store(smem, kq_off(false, jr, c0), rkv);
        tc::f16x8_store(smem, kq_off(true, jr, c0), rqv);
        tc::f16x8_store(rec, REC_KQ + tc::cm_offset(jr, c0, 128, KQ_SBO), kt);
        tc::f16x8_store(rec, REC_KQ + tc::cm_offset(C + jr, c0, 128, KQ_SBO), qt);
        tc::f16x8_store(smem, M::CD + tc::cm_offset(jr, c0, 128, tc::dense_sbo(D)), cd);
        // C_off(I, J) = k^ exp(G_ref(I) - G_j) / 256 = ke exp(G_ref(I) - G_end(J)) for every
        // later sub-block I (warp-uniform J): factor 1 for I = J + 1, F for I = J + 2, J + 3
        if (J < 3)
          tc::f16x8_store(smem, M::CO + tc::cm_offset(16 * off_slot(J + 1, J) + (jr & 15), c0, 128,
                                                      tc::dense_sbo(D)),
                          ke);
        if (J < 2) {
          float f[8], co[8];
          load8(f, sF + (J == 0 ? 0 : 2) * 128 + c0);      // (2, 0) or (3, 1)
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 x = mul2(make_float2(ke[e], ke[e + 1]), make_float2(f[e], f[e + 1]));
            co[e] = x.x;
            co[e + 1] = x.y;
          }
          tc::f16x8_store(smem, M::CO + tc::cm_offset(16 * off_slot(J + 2, J) + (jr & 15), c0, 128,
                                                      tc::dense_sbo(D)),
                          co);
        }
        if (J == 0) {
          float f[8], co[8];
          load8(f, sF + 128 + c0);                         // (3, 0)
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 x = mul2(make_float2(ke[e], ke[e + 1]), make_float2(f[e], f[e + 1]));
            co[e] = x.x;
            co[e + 1] = x.y;
          }
          tc::f16x8_store(smem, M::CO + tc::cm_offset(16 * off_slot(3, 0) + (jr & 15), c0, 128,
                                                      tc::dense_sbo(D)),
                          co);
        }
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------------------------------------------------------- A-GEMM
    // R C_diag^T (thread 0, N = 64, onto the exact pairs when there are any) and R C_off^T
    // (thread 32, N = 96); R is the swizzled K-major row operand, K steps of 32 bytes within
    // a 64-channel half
    if (tid == 0 || tid == 32) {
      const bool second = tid == 32;
      const uint32_t araw = tc::smem_u32(smem + M::RAW);
      auto dak = [&](int s) {
        return tc::desc_add(tc::smem_desc_sw128(araw + (s >> 2) * M::AK_HALF, 1024), (s & 3) * 32);
      };
      const uint64_t db = tc::smem_desc(tc::smem_u32(smem + (second ? M::CO : M::CD)), 128, tc::dense_sbo(D));
      const uint32_t id = tc::idesc_f16(128, second ? 96 : 64, tc::kF16);
      const uint32_t d = tmem + (second ? F_O : F_D);
      const uint32_t acc0 = (!second && s_anyslow) ? 1u : 0u;
#pragma unroll
      for (int s = 0; s < D / 16; ++s) tc::mma_ss(d, dak(s), tc::desc_add(db, s * 256), id, s > 0 ? 1u : acc0);
      tc::mma_commit(second ? &s_bar2 : &s_bar);
    }
    mma_wait2();
  } else {
    if (warp == 0) {                            // scalar: warp scan of 64 values
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
    if (tid < C) sKF[tid] *= sRK[tid];
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // A-GEMM [K; Q] K^T on the raw rows: two issuing threads (one issues a tcgen05.mma only
    // about every 100 cycles), one channel half each, the second into the X columns, which
    // are free until A has been extracted
    if (tid == 0 || tid == 32) {
      const bool second = tid == 32;
      const uint32_t id = tc::idesc_f16(128, 64, tc::kBF16);
      const uint32_t d = tmem + (second ? F_X : F_A);
      const uint64_t dak = tc::smem_desc_sw128(tc::smem_u32(smem + MS::AK) + (second ? MS::AK_HALF : 0u), 1024);
#pragma unroll
      for (int s = 0; s < D / 32; ++s)
        tc::mma_ss(d, tc::desc_add(dak, s * 32), tc::desc_add(dak, s * 32), id, s > 0);
      tc::mma_commit(second ? &s_bar2 : &s_bar);
    }
    mma_wait2();
  }

  // ------------------------------------------------------------------ A_kk, A_qk
  {
    const bool is_k = row < C;
    const int i = is_k ? row : row - C;
    float x[32];
    if constexpr (PERCH) {
      // rows of sub-blocks 2p (this warp's lanes 0-15) and 2p + 1 (lanes 16-31); for each
      // 16-column sub-block J of this thread's half: the diagonal products for J = I, the
      // off-diagonal ones for J < I, nothing for J > I (the loads are warp-collective, so
      // both sub-blocks' columns are loaded and each lane keeps its own)
      const int p = (warp & 3) & 1;
      const bool hi = ((i >> 4) & 1) != 0;
      const float ri = is_k ? sBeta[i] : 1.f;
      const int Ilo = 2 * p, Ihi = 2 * p + 1;
      auto src = [&](int J, int I) -> int {      // warp-uniform tensor-memory column, -1: none
        return J < I ? static_cast<int>(F_O) + 16 * off_slot(I, J) : (J == I ? static_cast<int>(F_D) + 16 * J : -1);
      };
      const int J0 = 2 * chalf, J1 = 2 * chalf + 1;
      const int s0l = src(J0, Ilo), s0h = src(J0, Ihi), s1l = src(J1, Ilo), s1h = src(J1, Ihi);
      uint32_t a0[16], b0[16], a1[16], b1[16];   // every load issued before one wait
      if (s0l >= 0) tc::tmem_ld16(tmem + lane_addr + static_cast<uint32_t>(s0l), a0);
      if (s0h >= 0) tc::tmem_ld16(tmem + lane_addr + static_cast<uint32_t>(s0h), b0);
      if (s1l >= 0) tc::tmem_ld16(tmem + lane_addr + static_cast<uint32_t>(s1l), a1);
      if (s1h >= 0) tc::tmem_ld16(tmem + lane_addr + static_cast<uint32_t>(s1h), b1);
      tc::tmem_wait_ld();
      const bool none0 = (hi ? s0h : s0l) < 0, none1 = (hi ? s1h : s1l) < 0;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        x[e] = none0 ? 0.f : __uint_as_float(hi ? b0[e] : a0[e]) * ri;
        x[16 + e] = none1 ? 0.f : __uint_as_float(hi ? b1[e] : a1[e]) * ri;
      }
    } else {
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
      const float ri = is_k ? sRK[i] * sBeta[i] : sRQ[i];
      if (s_anchored) {                         // exp(G_i - G_j) = E_i F_j
        const float rie = ri * sEA[i];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 kf = *reinterpret_cast<const float4*>(sKF + 32 * chalf + e);
          x[e] = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]) * rie * kf.x;
          x[e + 1] = __uint_as_float(e + 1 < 16 ? r0[e + 1] : r1[e - 15]) * rie * kf.y;
          x[e + 2] = __uint_as_float(e + 2 < 16 ? r0[e + 2] : r1[e - 14]) * rie * kf.z;
          x[e + 3] = __uint_as_float(e + 3 < 16 ? r0[e + 3] : r1[e - 13]) * rie * kf.w;
        }
      } else {                                  // exact per pair for extreme decays
        const float gi = sGs[i];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int j = 32 * chalf + e;
          x[e] = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]) * ri * sRK[j] * __expf(gi - sGs[j]);
        }
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
    float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float4 t = *reinterpret_cast<const float4*>(sT + sidx(c0 + m, c0 + c));
      const float2 am = make_float2(a[m], a[m]);
      acc01 = fma2(am, make_float2(t.x, t.y), acc01);
      acc23 = fma2(am, make_float2(t.z, t.w), acc23);
    }
    *reinterpret_cast<float4*>(sX + (16 * p + r) * XP + c) = make_float4(acc01.x, acc01.y, acc23.x, acc23.y);
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
    float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float4 x = *reinterpret_cast<const float4*>(sX + (16 * p + m) * XP + c);
      const float2 am = make_float2(a[m], a[m]);
      acc01 = fma2(am, make_float2(x.x, x.y), acc01);
      acc23 = fma2(am, make_float2(x.z, x.w), acc23);
    }
    *reinterpret_cast<float4*>(sT + sidx(r0 + r, c0 + c)) = make_float4(-acc01.x, -acc01.y, -acc23.x, -acc23.y);
  }
  __syncthreads();
  {                                             // X = A21 T11, one 32x32 pair
    // warp w: columns [4w, 4w + 4), lane: row; T11 is lower triangular, so rows m < 4w of it
    // are zero in these columns and the sum starts at the warp-uniform m = 4w
    const int r = lane, c = 4 * warp;
    float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
    float2 bcc01 = make_float2(0.f, 0.f), bcc23 = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int m = c; m < 32; m += 4) {
      const float4 av = *reinterpret_cast<const float4*>(sA + sidx(32 + r, m));
      const float4 t0 = *reinterpret_cast<const float4*>(sT + sidx(m, c));
      const float4 t1 = *reinterpret_cast<const float4*>(sT + sidx(m + 1, c));
      const float4 t2 = *reinterpret_cast<const float4*>(sT + sidx(m + 2, c));
      const float4 t3 = *reinterpret_cast<const float4*>(sT + sidx(m + 3, c));
      acc01 = fma2(make_float2(av.x, av.x), make_float2(t0.x, t0.y), acc01);
      acc23 = fma2(make_float2(av.x, av.x), make_float2(t0.z, t0.w), acc23);
      bcc01 = fma2(make_float2(av.y, av.y), make_float2(t1.x, t1.y), bcc01);
      bcc23 = fma2(make_float2(av.y, av.y), make_float2(t1.z, t1.w), bcc23);
      acc01 = fma2(make_float2(av.z, av.z), make_float2(t2.x, t2.y), acc01);
      acc23 = fma2(make_float2(av.z, av.z), make_float2(t2.z, t2.w), acc23);
      bcc01 = fma2(make_float2(av.w, av.w), make_float2(t3.x, t3.y), bcc01);
      bcc23 = fma2(make_float2(av.w, av.w), make_float2(t3.z, t3.w), bcc23);
    }
    acc01 = add2(acc01, bcc01);
    acc23 = add2(acc23, bcc23);
    *reinterpret_cast<float4*>(sX + r * XP + c) = make_float4(acc01.x, acc01.y, acc23.x, acc23.y);
  }
  __syncthreads();
  {                                             // T21 = -T22 X
    // warp w: rows [4w, 4w + 4); T22 is lower triangular, so the sum stops at m = 4w + 3
    const int r = tid >> 3, c = (tid & 7) * 4, mend = 4 * warp + 4;
    float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
    float2 bcc01 = make_float2(0.f, 0.f), bcc23 = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int m = 0; m < mend; m += 4) {
      const float4 av = *reinterpret_cast<const float4*>(sT + sidx(32 + r, 32 + m));
      const float4 x0 = *reinterpret_cast<const float4*>(sX + m * XP + c);
      const float4 x1 = *reinterpret_cast<const float4*>(sX + (m + 1) * XP + c);
      const float4 x2 = *reinterpret_cast<const float4*>(sX + (m + 2) * XP + c);
      const float4 x3 = *reinterpret_cast<const float4*>(sX + (m + 3) * XP + c);
      acc01 = fma2(make_float2(av.x, av.x), make_float2(x0.x, x0.y), acc01);
      acc23 = fma2(make_float2(av.x, av.x), make_float2(x0.z, x0.w), acc23);
      bcc01 = fma2(make_float2(av.y, av.y), make_float2(x1.x, x1.y), bcc01);
      bcc23 = fma2(make_float2(av.y, av.y), make_float2(x1.z, x1.w), bcc23);
      acc01 = fma2(make_float2(av.z, av.z), make_float2(x2.x, x2.y), acc01);
      acc23 = fma2(make_float2(av.z, av.z), make_float2(x2.z, x2.w), acc23);
      bcc01 = fma2(make_float2(av.w, av.w), make_float2(x3.x, x3.y), bcc01);
      bcc23 = fma2(make_float2(av.w, av.w), make_float2(x3.z, x3.w), bcc23);
    }
    acc01 = add2(acc01, bcc01);
    acc23 = add2(acc23, bcc23);
    *reinterpret_cast<float4*>(sT + sidx(32 + r, c)) = make_float4(-acc01.x, -acc01.y, -acc23.x, -acc23.y);
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
      tc::f16x8_store(smem, MS::KEA + tc::mn_offset(m, c0, KE_LBO, KE_SBO), x);
    }
  }
  if (!PERCH && tid < D) reinterpret_cast<float*>(rec + REC_GAM)[tid] = sGam[tid];
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) {
    const uint64_t dtb = tc::smem_desc(tc::smem_u32(smem + M::TBT), TB_LBO, TB_SBO);
    if constexpr (PERCH) {                      // K_end^T from tensor memory
      const uint32_t id = tc::idesc_f16(128, 64, tc::kF16, false, false, true);
#pragma unroll
      for (int s = 0; s < C / 16; ++s)
        tc::mma_ts(tmem + F_A, tmem + F_KE + s * 8, tc::desc_add(dtb, s * 2 * TB_LBO), id, s > 0);
    } else {
      const uint32_t id = tc::idesc_f16(128, 64, tc::kF16, false, true, true);
      const uint64_t dke = tc::smem_desc(tc::smem_u32(smem + MS::KEA), KE_LBO, KE_SBO);
#pragma unroll
      for (int s = 0; s < C / 16; ++s)
        tc::mma_ss(tmem + F_A, tc::desc_add(dke, s * 2 * KE_LBO), tc::desc_add(dtb, s * 2 * TB_LBO), id, s > 0);
    }
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

  if (PERCH && s_range && tid == 0) {           // outside the domain: the chain leaves this
    plan.skip[static_cast<int64_t>(ci.seq) * HV + h] = 1;   // (sequence, head) untouched
    raise_device_error(P.err, KDA_DEVERR_DECAY_RANGE);
  }
  if (s_abort) {                                // the phases that may have timed out
    if (tid == 0) plan.skip[static_cast<int64_t>(ci.seq) * HV + h] = 1;
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
  const int HV = P.HV;
  const SeqHeadTile cta = seq_head_tile(plan, HV, D / BV);
  const int b = cta.b, h = cta.h, vt = cta.vt;
  const uint32_t bos = P.offsets[b], eos = P.offsets[b + 1];
  // empty, or a chunk of it outside the tensor-core path's domain (the front kernel raised
  // the device error): o and the slot are left as they were
  if (eos <= bos || plan.skip[static_cast<int64_t>(b) * HV + h] != 0) return;
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
  // for the output warps' flags: they publish no data (an MMA seen complete through its
  // barrier, or tensor-memory reads fenced and synchronised before), and a CTA fence there
  // would wait for the previous chunk's o stores to global memory
  auto note_flag = [&](int* flag, int value) { *reinterpret_cast<volatile int*>(flag) = value; };
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
      if (dt == 0) {
        // one flag for the compute warps: V(q), Kb(q) and gamma(q) are in place, and the X MMA
        // of chunk q may start -- its [K~; Q~] has landed and the o rows of chunk q - 2, which
        // shared its X buffer, are out.  A failed wait stops the group at its next barrier.
        if (wait_bar(&s_kqa_bar[q % KQA_SLOTS], (q / KQA_SLOTS) & 1) &&
            (q < 2 || wait_flag(&s_o_free, static_cast<int>(q) - 1)))
          set_flag(&s_ready, static_cast<int>(q) + 1);
      }
      __syncwarp();
    }
    tc::cp_async_wait_all();
  } else if (warp >= W_OUT) {
    // ------------------------------------------------------------------ output warps
    const int dq = tid - NT - NTD - 64;         // 0..63: token row, TMEM lane 64 + dq
    float* op = reinterpret_cast<float*>(smem + CH_OST) + dq * OS;
    for (uint32_t c = 0; c < nchunks; ++c) {
      const bool bad = !wait_bar(&s_bar_o, c & 1);
      if (tc::named_sync_or(3, NTO, bad || aborted())) break;
      if (dq == 0) note_flag(&s_o_done, static_cast<int>(c) + 1);
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
      if (dq == 0) note_flag(&s_o_free, static_cast<int>(c) + 1);
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
        // ready(c + 1): [K~; Q~ | A1o](c) in place, X(c & 1) free, V(c) and Kb(c) in place
        bad = !wait_flag(&s_ready, static_cast<int>(c) + 1);
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
      __syncwarp();                             // the other lanes wait here, not beside the issuer
      if (extract) {                            // E' = V - K~ S over V's slot
        // V(c), Kb(c): the issuing threads saw ready(c + 1) above; the rest look while X runs
        if ((tid & 127) != 0) bad = bad || !wait_flag(&s_ready, static_cast<int>(c) + 1);
        bad = bad || !wait_bar(&s_bar_x, c & 1);
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
        __syncwarp();
      }
      // gamma(c): the E' threads saw ready(c + 1) above; the rest look while Kb E' runs
      if (!extract) bad = bad || !wait_flag(&s_ready, static_cast<int>(c) + 1);
      bad = bad || !wait_bar(&s_bar_s, c & 1);
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
  // two CTAs per SM: each prefetches for the CTA one full wave later (scalar decay), or half a
  // wave later (per-channel decay: measured 0.679 -> 0.674 ms on 2 x 16384 tokens, 32 heads,
  // against a full wave)
  const int ahead = PERCH ? sm_count() : 2 * sm_count();
  k<<<dim3(static_cast<unsigned>(plan_max_chunks(P)), P.HV), tcs::NT, bytes, st>>>(P, plan, recs, tmq, tmk, tmg,
                                                                                   ahead);
  return cudaGetLastError();
}

template <bool SBF16>
static cudaError_t launch_chain_t(const Problem& P, const PlanView& plan, const unsigned char* recs,
                                  cudaStream_t st) {
  auto k = tc_chain_kernel<SBF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(tcs::CH_BYTES));
  if (e != cudaSuccess) return e;
  const unsigned ctas = seq_head_tile_ctas(P, tcs::D / tcs::BV);
  if (ctas == 0) return cudaErrorInvalidConfiguration;
  k<<<ctas, tcs::NTC, tcs::CH_BYTES, st>>>(P, plan, recs);
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
