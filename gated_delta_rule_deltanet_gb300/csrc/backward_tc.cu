// backward_tc.cu -- the backward pass's contractions over the value dimension on Blackwell
// tensor cores, for d = 128 and chunks of 64.
//
// The chunk form's backward ("You Could Have Come Up With Kimi Delta Attention", sec. 6,
// differentiated by the chain rule; "From Attention to Learned Memory", sec. 3, for the
// linear-attention terms) needs, per (chunk, value head), five products whose contraction
// runs over the value dimension.  With S the state entering the chunk, dS' the gradient
// w.r.t. the state leaving it, E = T diag(beta) (V - K~ S) the chunk's corrected values,
// dO the output gradient and dY = T^T dE (each stored [rows][value]):
//
//   [dO; dY] S^T   rows 0-63: dQ~ = dO S^T          rows 64-127: dY S^T (dK~ = -diag(beta) dY S^T)
//   [dO; dY] E^T   rows 0-63: dM = dO E^T (lower)   rows 64-127: dY E^T (dA = -dY E^T, strictly lower)
//   dS' E^T        dK_end^T (key channel x token)
//
// plus dgamma_c = sum_v dS'_cv S_cv and the first term of dbeta,
// dY_i . (V - K~ S)_i = dY_i . V_i - K~_i . (dY S^T)_i.
//
// Every operand is K-major with the value dimension as K, which is how each matrix is
// stored, so TMA copies 32-value column blocks of them with the 128-byte swizzle straight
// into the operand layout of kind::tf32 MMAs: fp32 operands read with a 10-bit mantissa
// (the precision of the forward's fp16 operands) and fp32's exponent range, which the
// gradients need (their scale is the caller's).  The value dimension runs through a
// two-stage ring in four blocks; the three accumulators (256 tensor-memory columns) stay in
// tensor memory until the epilogue stages them in shared memory for coalesced stores.
#include "backward.cuh"
#include "tc_utils.cuh"
#include "tma_maps.cuh"

namespace kda {

namespace bvt {

constexpr int C = 64, D = 128, NT = 256;
// one stage: 32 value columns (128 bytes a row) of each operand, 1024-byte aligned blocks
constexpr uint32_t A_OFF = 0;          // [dO; dY]: 128 rows
constexpr uint32_t S_OFF = 16384;      // S: 128 key channels
constexpr uint32_t DS_OFF = 32768;     // dS': 128 key channels
constexpr uint32_t E_OFF = 49152;      // E: 64 tokens
constexpr uint32_t STAGE = 57344, DATA = 2 * STAGE;
constexpr uint32_t SMEM = DATA + 1024;                      // + alignment slack, control block in it
constexpr uint32_t T_QK = 0, T_MA = 128, T_KE = 192, COLS = 256;
constexpr int SP = 132;                                     // epilogue staging row (floats)
constexpr uint32_t kWaitLimit = 1u << 22;

struct Ctrl {
  uint64_t full[2];    // a stage's TMA copies landed
  uint64_t mdone[2];   // the MMAs reading a stage completed
  uint32_t tmem;
  int bad;             // a bounded wait gave up
  float br1[C];        // dY_i . V_i
};
constexpr uint32_t CTRL_BYTES = (sizeof(Ctrl) + 15) & ~15u;
static_assert(CTRL_BYTES <= 512, "control block fits the slack on one side of the data");
static_assert(2 * (SMEM + 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(D * SP * 4 + C * SP * 4 <= DATA && D * SP * 4 <= DATA, "epilogue staging fits the ring");

}  // namespace bvt

__global__ void __launch_bounds__(bvt::NT, 2)
    bwd_vc_tc_kernel(Problem P, BwdWorkspace ws, BwdArgs A,
                     const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dy,
                     const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_ds,
                     const __grid_constant__ CUtensorMap tm_e) {
  using namespace bvt;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzled blocks need a 1024-byte aligned base; the control block takes the slack
  // before it when that is large enough, else the slack after the data
  const uint32_t pad = (1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* const data = smem_raw + pad;
  Ctrl* const ctl = reinterpret_cast<Ctrl*>(pad >= CTRL_BYTES ? smem_raw : data + DATA);

  const int gc = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int plan_valid = ws.loc.plan.info[1], plan_chunks = ws.loc.plan.info[0];
  if (plan_valid == 0 || gc >= plan_chunks) return;
  const ChunkInfo ci = ws.loc.plan.chunks[gc];
  const int HV = P.HV, n = ci.n;
  const int64_t unit = static_cast<int64_t>(gc) * HV + h;
  const bool delta = !(P.flags & KDA_FLAG_NO_DELTA);
  const uint32_t sd = tc::smem_u32(data);

  // value columns [32 q, 32 q + 32) of the five operands into stage q & 1
  auto issue = [&](int q) {
    const uint32_t st = sd + static_cast<uint32_t>(q & 1) * STAGE;
    uint64_t* bar = &ctl->full[q & 1];
    tc::mbar_arrive_expect_tx(bar, STAGE);
    tc::tma_load_3d(st + A_OFF, &tm_do, 32 * q, h, static_cast<int32_t>(ci.t0), bar);
    tc::tma_load_2d(st + A_OFF + C * 128, &tm_dy, 32 * q, static_cast<int32_t>(unit * C), bar);
    tc::tma_load_2d(st + S_OFF, &tm_s, 32 * q, static_cast<int32_t>(unit * D), bar);
    tc::tma_load_2d(st + DS_OFF, &tm_ds, 32 * q, static_cast<int32_t>(unit * D), bar);
    tc::tma_load_2d(st + E_OFF, &tm_e, 32 * q, static_cast<int32_t>(unit * C), bar);
  };

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&ctl->full[s], 1);
      tc::mbar_init(&ctl->mdone[s], 1);
    }
    ctl->bad = 0;
    tc::fence_mbar_init();
    issue(0);
    issue(1);
  }
  if (warp == 0) {
    tc::tmem_alloc(&ctl->tmem, COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem;

  const uint32_t id_qk = tc::idesc_f16(128, 128, tc::kTF32);
  const uint32_t id_e = tc::idesc_f16(128, 64, tc::kTF32);
  // partial sums: dgamma of key channel tid / 2 (16 of each block's 32 values), dY_i . V_i
  // of token tid / 4 (8 values)
  float dg = 0.f, br = 0.f;
  const int gcr = tid >> 1, ghalf = tid & 1;
  const int bi = tid >> 2, bpart = tid & 3;
  const uint16_t* vrow = static_cast<const uint16_t*>(P.v) + (ci.t0 + bi) * P.v_stride +
                         static_cast<int64_t>(h) * D + 8 * bpart;

  for (int q = 0; q < 4; ++q) {
    const uint32_t st = static_cast<uint32_t>(q & 1);
    const uint32_t par = static_cast<uint32_t>(q >> 1) & 1u;
    const bool landed = tc::mbar_wait_bounded(&ctl->full[st], par, kWaitLimit);
    if (!landed) ctl->bad = 1;
    if (tid == 0 && landed) {
      tc::fence_after_sync();
      const uint32_t base = sd + st * STAGE;
      const uint64_t da = tc::smem_desc_sw128(base + A_OFF, 1024);
      const uint64_t ds = tc::smem_desc_sw128(base + S_OFF, 1024);
      const uint64_t dd = tc::smem_desc_sw128(base + DS_OFF, 1024);
      const uint64_t de = tc::smem_desc_sw128(base + E_OFF, 1024);
#pragma unroll
      for (int k = 0; k < 4; ++k) {             // K = 8 values (32 bytes) per instruction
        const uint32_t acc = (q > 0 || k > 0) ? 1u : 0u;
        tc::mma_ss_tf32(tmem + T_QK, tc::desc_add(da, 32 * k), tc::desc_add(ds, 32 * k), id_qk, acc);
        tc::mma_ss_tf32(tmem + T_MA, tc::desc_add(da, 32 * k), tc::desc_add(de, 32 * k), id_e, acc);
        tc::mma_ss_tf32(tmem + T_KE, tc::desc_add(dd, 32 * k), tc::desc_add(de, 32 * k), id_e, acc);
      }
      tc::mma_commit(&ctl->mdone[st]);
    }
    if (landed) {
      const unsigned char* blk = data + st * STAGE;
#pragma unroll
      for (int j = 0; j < 4; ++j) {             // S and dS' rows of key channel gcr
        const uint32_t off = tc::sw128_offset(gcr, 4 * ghalf + j);
        const float4 a = *reinterpret_cast<const float4*>(blk + S_OFF + off);
        const float4 b = *reinterpret_cast<const float4*>(blk + DS_OFF + off);
        dg += a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
      }
      if (bi < n) {                             // dY row bi (block rows 64-127) against V
        float vv[8];
        tc::bf16x8_load(reinterpret_cast<const unsigned char*>(vrow + 32 * q), vv);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float4 y = *reinterpret_cast<const float4*>(blk + A_OFF + tc::sw128_offset(C + bi, 2 * bpart + j));
          br += y.x * vv[4 * j] + y.y * vv[4 * j + 1] + y.z * vv[4 * j + 2] + y.w * vv[4 * j + 3];
        }
      }
    }
    __syncthreads();                            // the stage's shared-memory reads are done
    if (tid == 0 && q + 2 < 4) {
      if (tc::mbar_wait_bounded(&ctl->mdone[st], par, kWaitLimit)) issue(q + 2);
      else ctl->bad = 1;
    }
  }
  dg += __shfl_xor_sync(0xffffffffu, dg, 1);
  br += __shfl_xor_sync(0xffffffffu, br, 1);
  br += __shfl_xor_sync(0xffffffffu, br, 2);
  if (ghalf == 0) ws.dgam[unit * D + gcr] = dg;
  if (bpart == 0) ctl->br1[bi] = br;
  // the last commit covers every MMA of the CTA
  if (!tc::mbar_wait_bounded(&ctl->mdone[1], 1, kWaitLimit)) ctl->bad = 1;
  tc::fence_after_sync();
  __syncthreads();
  if (ctl->bad) {
    if (tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
  } else {
    float* stg = reinterpret_cast<float*>(data);   // the ring is free: staging rows of SP
    const int qd = warp & 3, ch = warp >> 2;
    const int r = 32 * qd + lane;                 // TMEM lane = accumulator row
    const uint32_t lane_addr = static_cast<uint32_t>(32 * qd) << 16;
    // [dO; dY] S^T: warp w reads lanes 32 (w % 4).. and columns 64 (w / 4)..
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      uint32_t v[16];
      tc::tmem_ld16(tmem + lane_addr + T_QK + 64 * ch + 16 * jj, v);
      tc::tmem_wait_ld();
      float* dst = stg + r * SP + 64 * ch + 16 * jj;
#pragma unroll
      for (int e = 0; e < 16; e += 4)
        *reinterpret_cast<float4*>(dst + e) = make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                                          __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
    }
    __syncthreads();
    // one warp per row: dQ~ (rows 0-63), dK~ = -diag(beta) dY S^T and dbeta's first term
    for (int rr = warp; rr < 2 * C; rr += NT / 32) {
      const float4 x = *reinterpret_cast<const float4*>(stg + rr * SP + 4 * lane);
      if (rr < C) {
        const float4 o = rr < n ? x : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(ws.dQt + (unit * C + rr) * D + 4 * lane) = o;
      } else {
        const int i = rr - C;
        const bool live = delta && i < n;
        const float nb = live ? -P.beta[(ci.t0 + i) * HV + h] : 0.f;
        *reinterpret_cast<float4*>(ws.dKt + (unit * C + i) * D + 4 * lane) =
            make_float4(nb * x.x, nb * x.y, nb * x.z, nb * x.w);
        float kd = 0.f;
        if (live) {
          const float4 kt = *reinterpret_cast<const float4*>(ws.loc.Kt + (unit * C + i) * D + 4 * lane);
          kd = kt.x * x.x + kt.y * x.y + kt.z * x.z + kt.w * x.w;
        }
        kd = warp_sum(kd);
        if (lane == 0) ws.dbr[unit * C + i] = i < n ? ctl->br1[i] - kd : 0.f;
      }
    }
    __syncthreads();
    // [dO; dY] E^T into the same rows; dS' E^T transposed to [token][key channel] after them
    float* stg2 = stg + 2 * C * SP;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      uint32_t v[16], w[16];
      tc::tmem_ld16(tmem + lane_addr + T_MA + 32 * ch + 16 * jj, v);
      tc::tmem_ld16(tmem + lane_addr + T_KE + 32 * ch + 16 * jj, w);
      tc::tmem_wait_ld();
      float* dst = stg + r * SP + 32 * ch + 16 * jj;
#pragma unroll
      for (int e = 0; e < 16; e += 4)
        *reinterpret_cast<float4*>(dst + e) = make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                                          __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
#pragma unroll
      for (int e = 0; e < 16; ++e) stg2[(32 * ch + 16 * jj + e) * SP + r] = __uint_as_float(w[e]);
    }
    __syncthreads();
    for (int rr = warp; rr < 2 * C; rr += NT / 32) {   // dM, dA: two tokens m per lane
      const float2 x = *reinterpret_cast<const float2*>(stg + rr * SP + 2 * lane);
      const int m = 2 * lane;
      if (rr < C) {
        const bool li = rr < n;
        *reinterpret_cast<float2*>(ws.dM + (unit * C + rr) * C + m) =
            make_float2(li && m <= rr ? x.x : 0.f, li && m + 1 <= rr ? x.y : 0.f);
      } else {
        const int i = rr - C;
        const bool li = delta && i < n;
        *reinterpret_cast<float2*>(ws.dA + (unit * C + i) * C + m) =
            make_float2(li && m < i ? -x.x : 0.f, li && m + 1 < i ? -x.y : 0.f);
      }
    }
    for (int m = warp; m < C; m += NT / 32)            // dK_end rows
      *reinterpret_cast<float4*>(ws.dKe + (unit * C + m) * D + 4 * lane) =
          *reinterpret_cast<const float4*>(stg2 + m * SP + 4 * lane);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, COLS);
}

cudaError_t launch_bwd_vc_tc(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A,
                             cudaStream_t st) {
  using namespace bvt;
  const int mc = plan_max_chunks(P);
  if (mc <= 0) return cudaSuccess;
  const uint64_t units = static_cast<uint64_t>(mc) * static_cast<uint64_t>(P.HV);
  alignas(64) CUtensorMap tdo, tdy, ts, tds, te;
  if (!encode_f32_token_blocks(&tdo, A.d_o, static_cast<uint64_t>(P.T), static_cast<uint64_t>(P.HV), D, C) ||
      !encode_f32_blocks(&tdy, ws.dY, units * C, D, D, C) || !encode_f32_blocks(&ts, ws.Sck, units * D, D, D, D) ||
      !encode_f32_blocks(&tds, ws.dSck, units * D, D, D, D) || !encode_f32_blocks(&te, ws.E, units * C, D, D, C))
    return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(bwd_vc_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM));
  if (e != cudaSuccess) return e;
  bwd_vc_tc_kernel<<<dim3(static_cast<unsigned>(mc), P.HV), NT, SMEM, st>>>(P, ws, A, tdo, tdy, ts, tds, te);
  return cudaGetLastError();
}

}  // namespace kda
