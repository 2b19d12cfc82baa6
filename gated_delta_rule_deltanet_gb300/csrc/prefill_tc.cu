// prefill_tc.cu -- chunkwise prefill on Blackwell tensor cores (tcgen05), d = 128, C = 64.
//
// One CTA owns one (sequence, value head, 64-wide value tile) and walks the
// sequence's chunks in order, keeping its 128 x 64 slice of the state in fp32
// registers.  Every contraction of the chunk form ("You Could Have Come Up With
// Kimi Delta Attention", sec. 6.3-6.5; "From Attention to Learned Memory",
// sec. 4, WY/UT transform and the 16x16 blocked inverse) runs as a tcgen05 MMA
// with fp32 accumulators in tensor memory:
//
//   A-GEMM   [K+; Q+] K-^T               -> A_kk (raw), A_qk (raw)      M=128 N=64  K=128
//            (scalar decay: raw bf16 q, k and exp(G_i - G_j) applied to the
//             result; per-channel decay: fp16 operands k exp(G - G_a),
//             q exp(G - G_a), k exp(G_a - G) with a mid-chunk anchor G_a)
//   solve    T = (I + A_kk)^-1 on CUDA cores (16x16 forward substitution,
//            then T21 = -T22 A21 T11 merges), TB = T diag(beta)
//   X        [I; A_qk] TB          = [TB; A_qk TB]                    M=128 N=64  K=64
//   Y        [TB; A_qk TB] K~      = [W; A_qk W],  K~ = k exp(G)      M=128 N=128 K=64
//   chain    [TB, -W; A_qk TB, Q~ - A_qk W] [V; S]  = [E; O]          M=128 N=64  K=192
//            K_end^T E  = dS,  S <- diag(gamma) S + dS               M=128 N=64  K=64
//
// (E = U - W S are the corrected values and O = Q~ S + A_qk E the outputs of the
// chunk; folding A_qk into the first operand gives O from the same MMA as E.)
// Operands are fp16 (10-bit mantissa, the same as tf32) except the raw bf16
// inputs of the scalar-decay A-GEMM; every value fed to them is bounded (decay
// factors <= 1, unit keys), so fp16 range is not a constraint.  Per-channel
// decay uses exp(G_i - G_a) and exp(G_a - G_j) with the anchor at the chunk's
// middle token, which keeps both factors finite while the cumulative decay over
// half a chunk stays below ~11 nats per channel.
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

// shared-memory map (bytes)
constexpr uint32_t S_K = 0;                    // k staging bf16 [64][128]
constexpr uint32_t S_Q = S_K + C * D * 2;      // q staging bf16 [64][128]
constexpr uint32_t S_V = S_Q + C * D * 2;      // v staging bf16 [64][64]
constexpr uint32_t S_G = S_V + C * BV * 2;     // log-decay -> cumulative G, fp32 [64][128]
constexpr uint32_t S_BETA = S_G + C * D * 4;   // beta [64]
constexpr uint32_t S_RK = S_BETA + 256;        // 1/|k| [64]
constexpr uint32_t S_RQ = S_RK + 256;          // scale/|q| [64]
constexpr uint32_t S_GAM = S_RQ + 256;         // exp(G_last) [128]
constexpr uint32_t S_GA = S_GAM + 512;         // anchor G_a [128]
constexpr uint32_t R1 = (S_GA + 512 + 1023) & ~1023u;
//   A-GEMM operands, then the chain's first operands
constexpr uint32_t AK = R1;                    // [K+; Q+] 128 x 128 (16-bit)
constexpr uint32_t BK = AK + 128 * 128 * 2;    // K- 64 x 128
constexpr uint32_t A1 = R1;                    // [TB; A_qk TB] 128 x 64 fp16
constexpr uint32_t A2 = A1 + 128 * 64 * 2;     // [-W; Q~ - A_qk W] 128 x 128 fp16
constexpr uint32_t R2 = BK + 64 * 128 * 2;
//   triangular solve, then K~^T and K_end^T
constexpr int SP = 65;                         // padded row of the fp32 solve tiles
constexpr uint32_t SOL_A = R2;                 // A_kk fp32 [64][65]
constexpr uint32_t SOL_T = SOL_A + C * SP * 4; // T fp32 [64][65]
constexpr uint32_t SOL_X = SOL_T + C * SP * 4; // merge temporaries fp32 [32][33]
constexpr uint32_t KTT = R2;                   // K~^T 128 x 64 fp16
constexpr uint32_t KET = KTT + 128 * 64 * 2;   // K_end^T 128 x 64 fp16
constexpr uint32_t R3 = (SOL_X + 32 * 33 * 4 + 127) & ~127u;
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
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// TMEM columns
constexpr uint32_t T_A = 0, T_X = 64, T_Y = 128, T_D1 = 256, T_D2 = 320, T_COLS = 512;

// dense K-major tiles: lbo 128, sbo = (K / 8) * 128
__host__ __device__ constexpr uint32_t dense_sbo(uint32_t K) { return (K / 8) * 128; }

__device__ __forceinline__ uint32_t f16x8_store(unsigned char* smem, uint32_t off, const float* x) {
  uint4 v;
  v.x = tc::pack_f16x2(x[0], x[1]);
  v.y = tc::pack_f16x2(x[2], x[3]);
  v.z = tc::pack_f16x2(x[4], x[5]);
  v.w = tc::pack_f16x2(x[6], x[7]);
  *reinterpret_cast<uint4*>(smem + off) = v;
  return 0;
}

__device__ __forceinline__ uint16_t f16_bits(float x) {
  return static_cast<uint16_t>(tc::pack_f16x2(x, 0.f) & 0xffffu);
}

__device__ __forceinline__ float bf16_at(const unsigned char* smem, uint32_t off, int idx) {
  return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(smem + off)[idx]);
}

}  // namespace tcp

template <bool PERCH, bool SBF16>
__global__ void __launch_bounds__(tcp::NT, 1) tc_prefill_kernel(Problem P, PlanView plan) {
  using namespace tcp;
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ uint64_t s_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (plan.info[1] == 0) return;
  const int b = blockIdx.x, h = blockIdx.y, vt = blockIdx.z;
  const int HV = P.HV;
  const int kh = h / (HV / P.HK);
  const uint32_t bos = P.offsets[b], eos = P.offsets[b + 1];
  if (eos <= bos) return;
  const int64_t sbase = (static_cast<int64_t>(P.slot_idx[b]) * HV + h) * D * D + vt * BV;

  float* sG = reinterpret_cast<float*>(smem + S_G);
  float* sBeta = reinterpret_cast<float*>(smem + S_BETA);
  float* sRK = reinterpret_cast<float*>(smem + S_RK);
  float* sRQ = reinterpret_cast<float*>(smem + S_RQ);
  float* sGam = reinterpret_cast<float*>(smem + S_GAM);
  float* sGA = reinterpret_cast<float*>(smem + S_GA);
  float* sA = reinterpret_cast<float*>(smem + SOL_A);
  float* sT = reinterpret_cast<float*>(smem + SOL_T);
  float* sX = reinterpret_cast<float*>(smem + SOL_X);

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

  // the fp32 master state: row `row` (key channel), value columns [32*chalf, +32)
  float S[32];
  {
    const int64_t base = sbase + static_cast<int64_t>(row) * D + 32 * chalf;
    for (int j = 0; j < 32; ++j)
      S[j] = SBF16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(P.pool)[base + j])
                   : static_cast<const float*>(P.pool)[base + j];
  }
  auto write_state_operand = [&]() {
    // S^T (N = value column j, K = key channel `row`), fp16, padded layout
    for (int j = 0; j < 32; ++j) {
      const int jj = 32 * chalf + j;
      *reinterpret_cast<uint16_t*>(smem + ST + tc::cm_offset(jj, row, LBO_P, ST_SBO)) = f16_bits(S[j]);
    }
  };
  write_state_operand();

  auto mma_wait = [&]() -> bool {
    const bool ok = tc::mbar_wait_bounded(&s_bar, phase & 1, kWaitLimit);
    phase ^= 1;
    if (!ok) s_abort = 1;
    tc::fence_after_sync();
    return ok;
  };

  const uint32_t nchunks = (eos - bos + C - 1) / C;
  for (uint32_t cidx = 0; cidx < nchunks; ++cidx) {
    const int64_t t0 = static_cast<int64_t>(bos) + static_cast<int64_t>(cidx) * C;
    const int n = static_cast<int>(min(static_cast<int64_t>(C), static_cast<int64_t>(eos) - t0));

    // ---------------------------------------------------------------- phase 0: load
    for (int u = tid; u < C * (D / 8); u += NT) {       // k, q rows: 16 vectors of 8 bf16
      const int i = u / (D / 8), q8 = u % (D / 8);
      uint4 kv = make_uint4(0, 0, 0, 0), qv = kv;
      if (i < n) {
        const int64_t t = t0 + i;
        kv = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(P.k) + t * P.k_stride +
                                             static_cast<int64_t>(kh) * D + q8 * 8);
        qv = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(P.q) + t * P.q_stride +
                                             static_cast<int64_t>(kh) * D + q8 * 8);
      }
      *reinterpret_cast<uint4*>(smem + S_K + (i * D + q8 * 8) * 2) = kv;
      *reinterpret_cast<uint4*>(smem + S_Q + (i * D + q8 * 8) * 2) = qv;
    }
    for (int u = tid; u < C * (BV / 8); u += NT) {
      const int i = u / (BV / 8), q8 = u % (BV / 8);
      uint4 vv = make_uint4(0, 0, 0, 0);
      if (i < n)
        vv = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(P.v) +
                                             (t0 + i) * P.v_stride + static_cast<int64_t>(h) * D +
                                             vt * BV + q8 * 8);
      *reinterpret_cast<uint4*>(smem + S_V + (i * BV + q8 * 8) * 2) = vv;
    }
    if (PERCH) {
      for (int u = tid; u < C * (D / 4); u += NT) {
        const int i = u / (D / 4), q4 = u % (D / 4);
        float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < n) gv = *reinterpret_cast<const float4*>(P.g + ((t0 + i) * HV + h) * D + q4 * 4);
        *reinterpret_cast<float4*>(sG + i * D + q4 * 4) = gv;
      }
    }
    for (int i = tid; i < C; i += NT) {
      const bool live = i < n;
      sBeta[i] = live ? P.beta[(t0 + i) * HV + h] : 0.f;
      if (!PERCH) sG[i] = live ? P.g[(t0 + i) * HV + h] : 0.f;
    }
    __syncthreads();

    // ---------------------------------------------------------------- phase 1: prep
    for (int i = warp; i < C; i += NT / 32) {
      float sk = 0.f, sq = 0.f;
      for (int c = lane; c < D; c += 32) {
        const float kx = bf16_at(smem, S_K, i * D + c), qx = bf16_at(smem, S_Q, i * D + c);
        sk += kx * kx;
        sq += qx * qx;
      }
      sk = warp_sum(sk);
      sq = warp_sum(sq);
      if (lane == 0) {
        sRK[i] = P.l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
        sRQ[i] = (P.l2norm ? rsqrtf(sq + 1e-6f) : 1.f) * P.scale;
      }
    }
    if (PERCH) {
      if (tid < D) {
        float acc = 0.f;
        for (int i = 0; i < C; ++i) {
          acc += sG[i * D + tid];
          sG[i * D + tid] = acc;
        }
        sGam[tid] = __expf(acc);
        sGA[tid] = sG[((n - 1) / 2) * D + tid];
      }
    } else if (tid == 0) {
      float acc = 0.f;
      for (int i = 0; i < C; ++i) {
        acc += sG[i];
        sG[i] = acc;
      }
      sGam[0] = __expf(acc);
    }
    __syncthreads();
    if (!PERCH) {
      if (tid < D) sGam[tid] = sGam[0];
      __syncthreads();
    }
    // A-GEMM operands: [K+; Q+] (rows 0-63 keys, 64-127 queries) and K-
    for (int u = tid; u < 3 * C * (D / 8); u += NT) {
      const int which = u / (C * (D / 8));          // 0: K+, 1: Q+, 2: K-
      const int r = (u / (D / 8)) % C, q8 = u % (D / 8);
      const uint32_t srcbase = which == 1 ? S_Q : S_K;
      const uint32_t src = srcbase + (r * D + q8 * 8) * 2;
      const uint32_t dst = which == 2 ? BK + tc::cm_offset(r, q8 * 8, 128, dense_sbo(D))
                                      : AK + tc::cm_offset(r + (which == 1 ? C : 0), q8 * 8, 128,
                                                           dense_sbo(D));
      if (!PERCH) {
        *reinterpret_cast<uint4*>(smem + dst) = *reinterpret_cast<const uint4*>(smem + src);
      } else {
        float x[8];
        for (int e = 0; e < 8; ++e) {
          const int c = q8 * 8 + e;
          const float gd = sG[r * D + c] - sGA[c];
          x[e] = bf16_at(smem, srcbase, r * D + c) * __expf(which == 2 ? -gd : gd);
        }
        f16x8_store(smem, dst, x);
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------------------------------------------------------- phase 2: A-GEMM
    if (tid == 0) {
      const uint32_t id = tc::idesc_f16(128, 64, PERCH ? tc::kF16 : tc::kBF16);
      for (int s = 0; s < D / 16; ++s)
        tc::mma_ss(tmem + T_A,
                   tc::smem_desc(tc::smem_u32(smem + AK) + s * 256, 128, dense_sbo(D)),
                   tc::smem_desc(tc::smem_u32(smem + BK) + s * 256, 128, dense_sbo(D)), id,
                   s > 0);
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
      const float ri = is_k ? sRK[i] * sBeta[i] : sRQ[i];
      float x[32];
      for (int e = 0; e < 32; ++e) {
        const int j = 32 * chalf + e;
        const float raw = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]);
        float a = raw * ri * sRK[j];
        if (!PERCH) a *= __expf(sG[i] - sG[j]);
        const bool keep = is_k ? (j < i) : (j <= i);
        x[e] = keep ? a : 0.f;
      }
      if (is_k) {
        for (int e = 0; e < 32; ++e) sA[i * SP + 32 * chalf + e] = x[e];
        // identity rows of L = [I; A_qk]
        float idv[32];
        for (int e = 0; e < 32; ++e) idv[e] = (32 * chalf + e == i) ? 1.f : 0.f;
        for (int g8 = 0; g8 < 4; ++g8)
          f16x8_store(smem, LMAT + tc::cm_offset(row, 32 * chalf + 8 * g8, 128, dense_sbo(64)),
                      idv + 8 * g8);
      } else {
        for (int g8 = 0; g8 < 4; ++g8)
          f16x8_store(smem, LMAT + tc::cm_offset(row, 32 * chalf + 8 * g8, 128, dense_sbo(64)),
                      x + 8 * g8);
      }
    }
    for (int idx = tid; idx < C * SP; idx += NT) sT[idx] = 0.f;
    tc::fence_before_sync();
    __syncthreads();

    // ---------------------------------------------------------------- phase 4: solve
    if (warp < C / 16 && lane < 16) {
      const int base = warp * 16, col = base + lane;
      for (int r = 0; r < 16; ++r) {
        const int rr = base + r;
        float val = r == lane ? 1.f : 0.f;
        for (int m = lane; m < r; ++m) val -= sA[rr * SP + base + m] * sT[(base + m) * SP + col];
        sT[rr * SP + col] = r >= lane ? val : 0.f;
        __syncwarp(0x0000ffffu);
      }
    }
    __syncthreads();
    for (int s = 16; s < C; s *= 2) {
      const int pairs = C / (2 * s);
      for (int idx = tid; idx < pairs * s * s; idx += NT) {
        const int p = idx / (s * s), r = (idx / s) % s, c = idx % s;
        const int r0 = 2 * p * s + s, c0 = 2 * p * s;
        float acc = 0.f;
        for (int m = c; m < s; ++m) acc += sA[(r0 + r) * SP + c0 + m] * sT[(c0 + m) * SP + c0 + c];
        sX[(p * s + r) * 33 + c] = acc;
      }
      __syncthreads();
      for (int idx = tid; idx < pairs * s * s; idx += NT) {
        const int p = idx / (s * s), r = (idx / s) % s, c = idx % s;
        const int r0 = 2 * p * s + s, c0 = 2 * p * s;
        float acc = 0.f;
        for (int m = 0; m <= r; ++m) acc += sT[(r0 + r) * SP + r0 + m] * sX[(p * s + m) * 33 + c];
        sT[(r0 + r) * SP + c0 + c] = -acc;
      }
      __syncthreads();
    }
    // TB^T[j][m] = T[m][j] beta_j  (N = j, K = m)
    for (int u = tid; u < C * (C / 8); u += NT) {
      const int j = u % C, m8 = u / C;
      float x[8];
      for (int e = 0; e < 8; ++e) x[e] = sT[(m8 * 8 + e) * SP + j] * sBeta[j];
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
      const float Gl = PERCH ? sG[(C - 1) * D + c] : sG[C - 1];
      float kt[8], ke[8];
      for (int e = 0; e < 8; ++e) {
        const int m = m8 * 8 + e;
        const float Gm = PERCH ? sG[m * D + c] : sG[m];
        const float kx = bf16_at(smem, S_K, m * D + c) * sRK[m];
        kt[e] = kx * __expf(Gm);
        ke[e] = kx * __expf(Gl - Gm);
      }
      f16x8_store(smem, KTT + tc::cm_offset(c, m8 * 8, 128, dense_sbo(64)), kt);
      f16x8_store(smem, KET + tc::cm_offset(c, m8 * 8, 128, dense_sbo(64)), ke);
    }
    for (int u = tid; u < BV * (C / 8); u += NT) {        // (value column j, 8 tokens)
      const int j = u % BV, m8 = u / BV;
      float x[8];
      for (int e = 0; e < 8; ++e) x[e] = bf16_at(smem, S_V, (m8 * 8 + e) * BV + j);
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
      for (int e = 0; e < 16; ++e) {
        x[e] = __uint_as_float(r0[e]);
        x[e + 16] = __uint_as_float(r1[e]);
      }
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
    for (int half = 0; half < 2; ++half) {
      const int c0 = 64 * chalf + 32 * half;
      uint32_t r0[16], r1[16];
      tc::tmem_ld16(tmem + lane_addr + T_Y + c0, r0);
      tc::tmem_ld16(tmem + lane_addr + T_Y + c0 + 16, r1);
      tc::tmem_wait_ld();
      float x[32];
      for (int e = 0; e < 32; ++e) {
        const float y = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]);
        float qt = 0.f;
        if (row >= C) {
          const int i = row - C, c = c0 + e;
          const float Gi = PERCH ? sG[i * D + c] : sG[i];
          qt = bf16_at(smem, S_Q, i * D + c) * sRQ[i] * __expf(Gi);
        }
        x[e] = qt - y;
      }
      for (int g8 = 0; g8 < 4; ++g8)
        f16x8_store(smem, A2 + tc::cm_offset(row, c0 + 8 * g8, 128, dense_sbo(D)), x + 8 * g8);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

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
        for (int e = 0; e < 32; ++e) {
          const float ev = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]);
          *reinterpret_cast<uint16_t*>(smem + ET + tc::cm_offset(32 * chalf + e, row, LBO_P, ET_SBO)) =
              f16_bits(ev);
        }
      } else if (row - C < n) {
        float* op = P.o + ((t0 + row - C) * HV + h) * D + vt * BV + 32 * chalf;
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
      uint32_t r0[16], r1[16];
      tc::tmem_ld16(tmem + lane_addr + T_D2 + 32 * chalf, r0);
      tc::tmem_ld16(tmem + lane_addr + T_D2 + 32 * chalf + 16, r1);
      tc::tmem_wait_ld();
      const float gam = sGam[row];
      for (int e = 0; e < 32; ++e)
        S[e] = gam * S[e] + __uint_as_float(e < 16 ? r0[e] : r1[e - 16]);
      write_state_operand();
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (s_abort) break;
  }

  if (s_abort) {
    // give the tensor core a last bounded chance to drain before TMEM is released
    tc::mbar_wait_bounded(&s_bar, phase & 1, kWaitLimit);
    if (tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
  } else {
    const int64_t base = sbase + static_cast<int64_t>(row) * D + 32 * chalf;
    for (int j = 0; j < 32; ++j) {
      if (SBF16)
        static_cast<uint16_t*>(P.pool)[base + j] = f32_to_bf16_bits(S[j]);
      else
        static_cast<float*>(P.pool)[base + j] = S[j];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, T_COLS);
}

bool tc_prefill_supported(const Problem& P, bool qbf16) {
  return qbf16 && P.D == tcp::D && P.chunk == tcp::C;
}

size_t tc_workspace_bytes(const Problem& P) { return plan_layout(P, nullptr, 0, nullptr); }

template <bool PERCH, bool SBF16>
static cudaError_t launch_tc_t(const Problem& P, const PlanView& plan, cudaStream_t st) {
  auto k = tc_prefill_kernel<PERCH, SBF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(tcp::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  k<<<dim3(P.num_seqs, P.HV, tcp::D / tcp::BV), tcp::NT, tcp::SMEM_BYTES, st>>>(P, plan);
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
  if (perch) e = sbf16 ? launch_tc_t<true, true>(P, plan, stream) : launch_tc_t<true, false>(P, plan, stream);
  else e = sbf16 ? launch_tc_t<false, true>(P, plan, stream) : launch_tc_t<false, false>(P, plan, stream);
  st.mark(2, stream);
  return e;
}

}  // namespace kda
