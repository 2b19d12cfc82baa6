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
// gradients need (their scale is the caller's).  The MMA reads only an operand's top bits,
// which would truncate every copied value toward zero, a bias that accumulates over a
// contraction; so every operand is rounded to the nearest tf32 first (in place after its
// copy here, where the threads write it in the scans).  The value dimension runs through a
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
                     const __grid_constant__ CUtensorMap tm_e, ChunkWindow win) {
  using namespace bvt;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzled blocks need a 1024-byte aligned base; the control block takes the slack
  // before it when that is large enough, else the slack after the data
  const uint32_t pad = (1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* const data = smem_raw + pad;
  Ctrl* const ctl = reinterpret_cast<Ctrl*>(pad >= CTRL_BYTES ? smem_raw : data + DATA);

  const int slot = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int gc;
  if (ws.loc.plan.info[1] == 0 || !window_chunk(ws.loc.plan, P.num_seqs, win, slot, &gc)) return;
  const ChunkInfo ci = ws.loc.plan.chunks[gc];
  const int HV = P.HV, n = ci.n;
  const int64_t unit = static_cast<int64_t>(slot) * HV + h;
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
    if (landed) {
      unsigned char* blk = data + st * STAGE;
      // the partial sums from the copied fp32 values ...
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
      __syncthreads();
      // ... then every value rounded to tf32 in place for the MMAs
      float4* b4 = reinterpret_cast<float4*>(blk);
      for (int u = tid; u < static_cast<int>(STAGE / 16); u += NT) {
        float4 x = b4[u];
        x.x = tf32_nearest(x.x);
        x.y = tf32_nearest(x.y);
        x.z = tf32_nearest(x.z);
        x.w = tf32_nearest(x.w);
        b4[u] = x;
      }
    } else {
      __syncthreads();
    }
    tc::fence_async_smem();
    __syncthreads();                            // the stage's shared-memory traffic is done
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

// ------------------------------------------------------------------------------- scans
//
// The state recursion and its transpose, per (sequence, value head, 64 value columns), chunk
// by chunk on tensor cores (kind::tf32).  Every operand is K-major: the local stage's matrices
// come from the workspace in the orientation each product needs (W and K_end as stored;
// K_end^T, Q~^T, W^T, A_qk^T and T^T as transposed copies), copied by TMA in 32-column blocks
// with the 128-byte swizzle; the running state and the per-chunk right-hand sides are written
// by the threads transposed (value rows, K = key channel or token) into the same layout.
//
//   forward   X = W S,  E = U - X,  S <- diag(gamma) S + K_end^T E
//   reverse   dE = A_qk^T dO + K_end dS',  dY = T^T dE,  dV = diag(beta) dY,
//             dS = diag(gamma) dS' + Q~^T dO - W^T dE
//
// Products with 64 rows (tokens) run as M = 128 MMAs whose rows 64-127 read the next block
// of shared memory: those accumulator lanes are never read.  Threads: warp w serves tensor-
// memory lanes 32 (w % 4).. and value columns 32 (w / 4).. of the 64-column accumulators, and
// keeps that 32-column row segment of the state (thread = key channel) in registers.

namespace bst {

constexpr int C = 64, D = 128, BV = 64, NT = 256;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint32_t BLK = 8192;                  // a 32-column block of 64 rows (128 B a row)
// forward: W (4 blocks + 8 KB under the last M = 128 read), K_end^T (2 blocks of 128 rows),
// U (2 blocks: the CTA's 64 value columns), S^T (4 blocks of 64 value rows), E^T (2 blocks)
constexpr uint32_t F_W = 0, F_KT = 5 * BLK, F_U = F_KT + 4 * BLK, F_ST = F_U + 2 * BLK,
                   F_ET = F_ST + 4 * BLK, F_DATA = F_ET + 2 * BLK;
// reverse: K_end (4 blocks), A_qk^T (2), T^T (2) + 8 KB, Q~^T and W^T (2 blocks of 128 rows
// each), dO^T (2 blocks of 64 value rows), dS'^T (4), dE^T (2)
constexpr uint32_t R_KE = 0, R_AQ = 4 * BLK, R_TT = 6 * BLK, R_QT = 9 * BLK, R_WT = R_QT + 4 * BLK,
                   R_OT = R_WT + 4 * BLK, R_RT = R_OT + 2 * BLK, R_ET = R_RT + 4 * BLK,
                   R_DATA = R_ET + 2 * BLK;
constexpr uint32_t F_BYTES_A = 4 * BLK + 2 * BLK, F_BYTES_B = 4 * BLK;   // W + U, K_end^T
constexpr uint32_t R_BYTES_A = 4 * BLK + 2 * BLK + 4 * BLK, R_BYTES_B = 2 * BLK + 4 * BLK;
static_assert(F_DATA + 1024 <= 227 * 1024 && R_DATA + 1024 <= 227 * 1024, "shared memory budget");

struct Ctrl {
  uint64_t full_a, full_b;   // the two TMA groups of a chunk
  uint64_t bar1, bar2;       // the two MMA groups of a chunk
  uint32_t tmem;
  int bad;
};
constexpr uint32_t CTRL_BYTES = (sizeof(Ctrl) + 15) & ~15u;

// byte offset of element (row, k) of a K-major operand stored as 32-column blocks of
// `rows_per_block` rows (128 bytes a row, 128-byte swizzle)
__device__ __forceinline__ uint32_t kmaj(uint32_t row, uint32_t k, uint32_t rows_per_block) {
  return (k >> 5) * rows_per_block * 128 + tc::sw128_offset(row, (k & 31) >> 2) + (k & 3) * 4;
}

}  // namespace bst

template <bool SBF16>
__global__ void __launch_bounds__(bst::NT, 1)
    bwd_fwd_scan_tc_kernel(Problem P, BwdWorkspace ws, const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_kt,
                           ChunkWindow win, int record) {
  using namespace bst;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* const data = smem_raw + pad;
  Ctrl* const ctl = reinterpret_cast<Ctrl*>(pad >= CTRL_BYTES ? smem_raw : data + F_DATA);
  if (ws.loc.plan.info[1] == 0) return;
  const SeqHeadTile cta = seq_head_tile(ws.loc.plan, P.HV, D / BV);
  const int b = cta.b, h = cta.h, v0 = cta.vt * BV;
  const int HV = P.HV, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this CTA's chunks: the sequence's, or those of window win.w (slots b * wc ..)
  const int c0 = ws.loc.plan.seq_chunk0[b], nb = ws.loc.plan.seq_chunk0[b + 1] - c0;
  const int j0 = win.wc ? win.w * win.wc : 0, j1 = win.wc ? min(nb, j0 + win.wc) : nb;
  if (j0 >= j1) return;
  const int first = c0 + j0, last = c0 + j1;
  const int slot0 = win.wc ? b * win.wc - first : 0;   // slot of chunk cidx: slot0 + cidx
  const int qd = warp & 3, chalf = warp >> 2;
  const int r = 32 * qd + lane;                 // TMEM lane: key channel (state) / token (X)
  const int vc = 32 * chalf;                    // this thread's 32 value columns within the tile
  const uint32_t lane_addr = static_cast<uint32_t>(32 * qd) << 16;
  const uint32_t sd = tc::smem_u32(data);
  auto unit_of = [&](int cidx) { return static_cast<int64_t>(slot0 + cidx) * HV + h; };

  auto load_a = [&](int cidx) {                 // W and the CTA's U columns of chunk cidx
    const int32_t row = static_cast<int32_t>(unit_of(cidx) * C);
    tc::mbar_arrive_expect_tx(&ctl->full_a, F_BYTES_A);
#pragma unroll
    for (int j = 0; j < 4; ++j) tc::tma_load_2d(sd + F_W + j * BLK, &tm_w, 32 * j, row, &ctl->full_a);
#pragma unroll
    for (int j = 0; j < 2; ++j) tc::tma_load_2d(sd + F_U + j * BLK, &tm_u, v0 + 32 * j, row, &ctl->full_a);
  };
  auto load_b = [&](int cidx) {                 // K_end^T of chunk cidx
    const int32_t row = static_cast<int32_t>(unit_of(cidx) * D);
    tc::mbar_arrive_expect_tx(&ctl->full_b, F_BYTES_B);
#pragma unroll
    for (int j = 0; j < 2; ++j) tc::tma_load_2d(sd + F_KT + j * 2 * BLK, &tm_kt, 32 * j, row, &ctl->full_b);
  };
  if (tid == 0) {
    tc::mbar_init(&ctl->full_a, 1);
    tc::mbar_init(&ctl->full_b, 1);
    tc::mbar_init(&ctl->bar1, 1);
    tc::mbar_init(&ctl->bar2, 1);
    ctl->bad = 0;
    tc::fence_mbar_init();
    load_a(first);
    load_b(first);
  }
  if (warp == 0) {
    tc::tmem_alloc(&ctl->tmem, 128);
    tc::tmem_relinquish();
  }
  float Sv[32];
  const int64_t sbase = (static_cast<int64_t>(P.slot_idx[b]) * HV + h) * D * D + static_cast<int64_t>(r) * D + v0 + vc;
  const int64_t row_off = static_cast<int64_t>(r) * D + v0 + vc;
  if (j0 > 0) {                                 // a later window: from its checkpoint
    const float* ck = ws.ckpt + (ckpt_entry(c0, win) * HV + h) * D * D + row_off;
#pragma unroll
    for (int j = 0; j < 32; ++j) Sv[j] = ck[j];
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      Sv[j] = SBF16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(P.pool)[sbase + j])
                    : static_cast<const float*>(P.pool)[sbase + j];
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem;
  constexpr uint32_t T_X = 0, T_D = 64;
  const uint32_t id = tc::idesc_f16(128, BV, tc::kTF32);

  for (int cidx = first; cidx < last; ++cidx) {
    const uint32_t par = static_cast<uint32_t>(cidx - first) & 1u;
    const int64_t unit = unit_of(cidx);
    const float gm = __ldg(ws.loc.gamma + unit * D + r);   // read at the update, issued now
    // S entering the chunk: into the workspace, and transposed as the B operand of W S
    {
      if (record) {
        float* gs = ws.Sck + (unit * D + r) * D + v0 + vc;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(gs + j) = make_float4(Sv[j], Sv[j + 1], Sv[j + 2], Sv[j + 3]);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) *reinterpret_cast<float*>(data + F_ST + kmaj(vc + j, r, 64)) = tf32_nearest(Sv[j]);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      if (tc::mbar_wait_bounded(&ctl->full_a, par, kWaitLimit)) {
        tc::fence_after_sync();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t da = tc::smem_desc_sw128(sd + F_W + j * BLK, 1024);
          const uint64_t db = tc::smem_desc_sw128(sd + F_ST + j * BLK, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_ss_tf32(tmem + T_X, tc::desc_add(da, 32 * k), tc::desc_add(db, 32 * k), id, (j | k) ? 1u : 0u);
        }
      } else {
        ctl->bad = 1;
      }
      tc::mma_commit(&ctl->bar1);
    }
    // E = U - X on the token rows (lanes 0-63), stored and written transposed
    const bool ok1 = tc::mbar_wait_bounded(&ctl->bar1, par, kWaitLimit) &&
                     tc::mbar_wait_bounded(&ctl->full_a, par, kWaitLimit);
    tc::fence_after_sync();
    if (!ok1) ctl->bad = 1;
    if (qd < 2) {
      uint32_t x0[16], x1[16];
      tc::tmem_ld16(tmem + lane_addr + T_X + vc, x0);
      tc::tmem_ld16(tmem + lane_addr + T_X + vc + 16, x1);
      tc::tmem_wait_ld();
      float e[32];
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 u = *reinterpret_cast<const float4*>(data + F_U + kmaj(r, vc + j, 64));
        const uint32_t* x = j < 16 ? x0 + j : x1 + (j - 16);
        e[j] = u.x - __uint_as_float(x[0]);
        e[j + 1] = u.y - __uint_as_float(x[1]);
        e[j + 2] = u.z - __uint_as_float(x[2]);
        e[j + 3] = u.w - __uint_as_float(x[3]);
      }
      if (record) {
        float* ge = ws.E + (unit * C + r) * D + v0 + vc;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(ge + j) = make_float4(e[j], e[j + 1], e[j + 2], e[j + 3]);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) *reinterpret_cast<float*>(data + F_ET + kmaj(vc + j, r, 64)) = tf32_nearest(e[j]);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      if (cidx + 1 < last) load_a(cidx + 1);    // W and U of this chunk are consumed
      if (tc::mbar_wait_bounded(&ctl->full_b, par, kWaitLimit)) {
        tc::fence_after_sync();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint64_t da = tc::smem_desc_sw128(sd + F_KT + j * 2 * BLK, 1024);
          const uint64_t db = tc::smem_desc_sw128(sd + F_ET + j * BLK, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_ss_tf32(tmem + T_D, tc::desc_add(da, 32 * k), tc::desc_add(db, 32 * k), id, (j | k) ? 1u : 0u);
        }
      } else {
        ctl->bad = 1;
      }
      tc::mma_commit(&ctl->bar2);
    }
    // S <- diag(gamma) S + K_end^T E
    const bool ok2 = tc::mbar_wait_bounded(&ctl->bar2, par, kWaitLimit);
    tc::fence_after_sync();
    if (!ok2) ctl->bad = 1;
    {
      uint32_t d0[16], d1[16];
      tc::tmem_ld16(tmem + lane_addr + T_D + vc, d0);
      tc::tmem_ld16(tmem + lane_addr + T_D + vc + 16, d1);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        Sv[j] = fmaf(gm, Sv[j], __uint_as_float(d0[j]));
        Sv[16 + j] = fmaf(gm, Sv[16 + j], __uint_as_float(d1[j]));
      }
    }
    if (tid == 0 && cidx + 1 < last) load_b(cidx + 1);   // K_end^T of this chunk is consumed
    if (tc::named_sync_or(1, NT, ctl->bad != 0)) break;
  }
  if (ctl->bad) {
    if (tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
  } else if (!record && j1 < nb) {              // the checkpoint of the next window
    ChunkWindow next = win;
    next.w += 1;
    float* ck = ws.ckpt + (ckpt_entry(c0, next) * HV + h) * D * D + row_off;
#pragma unroll
    for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(ck + j) = make_float4(Sv[j], Sv[j + 1], Sv[j + 2], Sv[j + 3]);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

__global__ void __launch_bounds__(bst::NT, 1)
    bwd_rev_scan_tc_kernel(Problem P, BwdWorkspace ws, BwdArgs A, const __grid_constant__ CUtensorMap tm_ke,
                           const __grid_constant__ CUtensorMap tm_aq, const __grid_constant__ CUtensorMap tm_qt,
                           const __grid_constant__ CUtensorMap tm_tt, const __grid_constant__ CUtensorMap tm_wt,
                           ChunkWindow win) {
  using namespace bst;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* const data = smem_raw + pad;
  Ctrl* const ctl = reinterpret_cast<Ctrl*>(pad >= CTRL_BYTES ? smem_raw : data + R_DATA);
  if (ws.loc.plan.info[1] == 0) return;
  const SeqHeadTile cta = seq_head_tile(ws.loc.plan, P.HV, D / BV);
  const int b = cta.b, h = cta.h, v0 = cta.vt * BV;
  const int HV = P.HV, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c0 = ws.loc.plan.seq_chunk0[b], nb = ws.loc.plan.seq_chunk0[b + 1] - c0;
  const int j0 = win.wc ? win.w * win.wc : 0, j1 = win.wc ? min(nb, j0 + win.wc) : nb;
  const int qd = warp & 3, chalf = warp >> 2;
  const int r = 32 * qd + lane;                 // TMEM lane: key channel (dS) / token (dE, dY)
  const int vc = 32 * chalf;
  const uint32_t lane_addr = static_cast<uint32_t>(32 * qd) << 16;
  const uint32_t sd = tc::smem_u32(data);
  const int64_t sbase = (static_cast<int64_t>(P.slot_idx[b]) * HV + h) * D * D + static_cast<int64_t>(r) * D + v0 + vc;
  float* const carry = ws.carry + (static_cast<int64_t>(b) * HV + h) * D * D + static_cast<int64_t>(r) * D + v0 + vc;
  if (j0 >= j1) {                               // no chunk here; an empty sequence: dS0 = dS_final
    if (nb == 0 && A.d_state0)
#pragma unroll
      for (int j = 0; j < 32; ++j) A.d_state0[sbase + j] = A.d_state ? A.d_state[sbase + j] : 0.f;
    return;
  }
  const int first = c0 + j0, last = c0 + j1;
  const int slot0 = win.wc ? b * win.wc - first : 0;
  // dS starts as the gradient w.r.t. the final state, or what the later window handed on
  float Rv[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) Rv[j] = j1 < nb ? carry[j] : (A.d_state ? A.d_state[sbase + j] : 0.f);
  auto unit_of = [&](int cidx) { return static_cast<int64_t>(slot0 + cidx) * HV + h; };
  auto load_a = [&](int cidx) {                 // K_end, A_qk^T, Q~^T of chunk cidx
    const int64_t u = unit_of(cidx);
    tc::mbar_arrive_expect_tx(&ctl->full_a, R_BYTES_A);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      tc::tma_load_2d(sd + R_KE + j * BLK, &tm_ke, 32 * j, static_cast<int32_t>(u * C), &ctl->full_a);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      tc::tma_load_2d(sd + R_AQ + j * BLK, &tm_aq, 32 * j, static_cast<int32_t>(u * C), &ctl->full_a);
      tc::tma_load_2d(sd + R_QT + j * 2 * BLK, &tm_qt, 32 * j, static_cast<int32_t>(u * D), &ctl->full_a);
    }
  };
  auto load_b = [&](int cidx) {                 // T^T, W^T of chunk cidx
    const int64_t u = unit_of(cidx);
    tc::mbar_arrive_expect_tx(&ctl->full_b, R_BYTES_B);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      tc::tma_load_2d(sd + R_TT + j * BLK, &tm_tt, 32 * j, static_cast<int32_t>(u * C), &ctl->full_b);
      tc::tma_load_2d(sd + R_WT + j * 2 * BLK, &tm_wt, 32 * j, static_cast<int32_t>(u * D), &ctl->full_b);
    }
  };
  if (tid == 0) {
    tc::mbar_init(&ctl->full_a, 1);
    tc::mbar_init(&ctl->full_b, 1);
    tc::mbar_init(&ctl->bar1, 1);
    tc::mbar_init(&ctl->bar2, 1);
    ctl->bad = 0;
    tc::fence_mbar_init();
    load_a(last - 1);
    load_b(last - 1);
  }
  if (warp == 0) {
    tc::tmem_alloc(&ctl->tmem, 256);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem;
  constexpr uint32_t T_DE = 0, T_DY = 64, T_DS = 128;
  const uint32_t id = tc::idesc_f16(128, BV, tc::kTF32);
  const int om = tid >> 2, opart = tid & 3;     // dO staging: token om, values 16 opart..
  // the next chunk's dO row segment, gamma and beta are loaded one chunk ahead
  float4 onext[4];
  auto load_do = [&](const ChunkInfo& c) {
    const float* src = A.d_o + ((c.t0 + om) * HV + h) * D + v0 + 16 * opart;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      onext[j] = om < c.n ? *reinterpret_cast<const float4*>(src + 4 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  ChunkInfo cnext = ws.loc.plan.chunks[last - 1];
  load_do(cnext);
  float gnext = __ldg(ws.loc.gamma + unit_of(last - 1) * D + r);
  float bnext = r < cnext.n ? P.beta[(cnext.t0 + r) * HV + h] : 0.f;

  for (int cidx = last - 1; cidx >= first; --cidx) {
    const uint32_t par = static_cast<uint32_t>(last - 1 - cidx) & 1u;
    const int64_t unit = unit_of(cidx);
    const ChunkInfo ci = cnext;
    const float gm = gnext, bt = bnext;
    // dO^T (rows past the chunk's end zero) and dS'^T as B operands; dS' into the workspace
    {
      float o[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o[4 * j] = onext[j].x; o[4 * j + 1] = onext[j].y; o[4 * j + 2] = onext[j].z; o[4 * j + 3] = onext[j].w;
      }
      if (cidx > first) {
        cnext = ws.loc.plan.chunks[cidx - 1];
        load_do(cnext);
        gnext = __ldg(ws.loc.gamma + unit_of(cidx - 1) * D + r);
        bnext = r < cnext.n ? P.beta[(cnext.t0 + r) * HV + h] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) *reinterpret_cast<float*>(data + R_OT + kmaj(16 * opart + j, om, 64)) = tf32_nearest(o[j]);
      float* gs = ws.dSck + (unit * D + r) * D + v0 + vc;
#pragma unroll
      for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(gs + j) = make_float4(Rv[j], Rv[j + 1], Rv[j + 2], Rv[j + 3]);
#pragma unroll
      for (int j = 0; j < 32; ++j) *reinterpret_cast<float*>(data + R_RT + kmaj(vc + j, r, 64)) = tf32_nearest(Rv[j]);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      if (tc::mbar_wait_bounded(&ctl->full_a, par, kWaitLimit)) {
        tc::fence_after_sync();
        // dE = A_qk^T dO + K_end dS'  (rows 0-63);  dS = Q~^T dO  (the rest after dE)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint64_t da = tc::smem_desc_sw128(sd + R_AQ + j * BLK, 1024);
          const uint64_t dq = tc::smem_desc_sw128(sd + R_QT + j * 2 * BLK, 1024);
          const uint64_t db = tc::smem_desc_sw128(sd + R_OT + j * BLK, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            tc::mma_ss_tf32(tmem + T_DE, tc::desc_add(da, 32 * k), tc::desc_add(db, 32 * k), id, (j | k) ? 1u : 0u);
            tc::mma_ss_tf32(tmem + T_DS, tc::desc_add(dq, 32 * k), tc::desc_add(db, 32 * k), id, (j | k) ? 1u : 0u);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t da = tc::smem_desc_sw128(sd + R_KE + j * BLK, 1024);
          const uint64_t db = tc::smem_desc_sw128(sd + R_RT + j * BLK, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_ss_tf32(tmem + T_DE, tc::desc_add(da, 32 * k), tc::desc_add(db, 32 * k), id, 1u);
        }
      } else {
        ctl->bad = 1;
      }
      tc::mma_commit(&ctl->bar1);
    }
    // -dE^T as the B operand of T^T dE and W^T dE (the sign folded into the operand, so both
    // products accumulate: dS gets + W^T (-dE), and T^T (-dE) = -dY)
    const bool ok1 = tc::mbar_wait_bounded(&ctl->bar1, par, kWaitLimit);
    tc::fence_after_sync();
    if (!ok1) ctl->bad = 1;
    if (qd < 2) {
      uint32_t x0[16], x1[16];
      tc::tmem_ld16(tmem + lane_addr + T_DE + vc, x0);
      tc::tmem_ld16(tmem + lane_addr + T_DE + vc + 16, x1);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        *reinterpret_cast<float*>(data + R_ET + kmaj(vc + j, r, 64)) = tf32_nearest(-__uint_as_float(x0[j]));
        *reinterpret_cast<float*>(data + R_ET + kmaj(vc + 16 + j, r, 64)) = tf32_nearest(-__uint_as_float(x1[j]));
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      if (cidx > first) load_a(cidx - 1);       // K_end, A_qk^T, Q~^T and dO^T are consumed
      if (tc::mbar_wait_bounded(&ctl->full_b, par, kWaitLimit)) {
        tc::fence_after_sync();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint64_t dt = tc::smem_desc_sw128(sd + R_TT + j * BLK, 1024);
          const uint64_t dw = tc::smem_desc_sw128(sd + R_WT + j * 2 * BLK, 1024);
          const uint64_t db = tc::smem_desc_sw128(sd + R_ET + j * BLK, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            tc::mma_ss_tf32(tmem + T_DY, tc::desc_add(dt, 32 * k), tc::desc_add(db, 32 * k), id, (j | k) ? 1u : 0u);
            tc::mma_ss_tf32(tmem + T_DS, tc::desc_add(dw, 32 * k), tc::desc_add(db, 32 * k), id, 1u);
          }
        }
      } else {
        ctl->bad = 1;
      }
      tc::mma_commit(&ctl->bar2);
    }
    // dY and dV on the token rows; dS = diag(gamma) dS' + (Q~^T dO - W^T dE) on every row
    const bool ok2 = tc::mbar_wait_bounded(&ctl->bar2, par, kWaitLimit);
    tc::fence_after_sync();
    if (!ok2) ctl->bad = 1;
    if (qd < 2) {
      uint32_t y0[16], y1[16];
      tc::tmem_ld16(tmem + lane_addr + T_DY + vc, y0);
      tc::tmem_ld16(tmem + lane_addr + T_DY + vc + 16, y1);
      tc::tmem_wait_ld();
      float y[32];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        y[j] = -__uint_as_float(y0[j]);
        y[16 + j] = -__uint_as_float(y1[j]);
      }
      float* gy = ws.dY + (unit * C + r) * D + v0 + vc;
#pragma unroll
      for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(gy + j) = make_float4(y[j], y[j + 1], y[j + 2], y[j + 3]);
      if (r < ci.n) {
        float* gv = A.dv + ((ci.t0 + r) * HV + h) * D + v0 + vc;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(gv + j) = make_float4(bt * y[j], bt * y[j + 1], bt * y[j + 2], bt * y[j + 3]);
      }
    }
    {
      uint32_t d0[16], d1[16];
      tc::tmem_ld16(tmem + lane_addr + T_DS + vc, d0);
      tc::tmem_ld16(tmem + lane_addr + T_DS + vc + 16, d1);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        Rv[j] = fmaf(gm, Rv[j], __uint_as_float(d0[j]));
        Rv[16 + j] = fmaf(gm, Rv[16 + j], __uint_as_float(d1[j]));
      }
    }
    if (tid == 0 && cidx > first) load_b(cidx - 1);     // T^T and W^T of this chunk are consumed
    if (tc::named_sync_or(1, NT, ctl->bad != 0)) break;
  }
  if (ctl->bad) {
    if (tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
  } else if (j0 > 0) {                          // handed to the earlier window
#pragma unroll
    for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(carry + j) = make_float4(Rv[j], Rv[j + 1], Rv[j + 2], Rv[j + 3]);
  } else if (A.d_state0) {
#pragma unroll
    for (int j = 0; j < 32; ++j) A.d_state0[sbase + j] = Rv[j];
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

cudaError_t launch_bwd_scans_tc(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A, bool sbf16,
                                ChunkWindow win, int slots, bool record, cudaStream_t st) {
  using namespace bst;
  const uint64_t units = static_cast<uint64_t>(slots > 0 ? slots : 1) * static_cast<uint64_t>(P.HV);
  alignas(64) CUtensorMap tw, tu, tkt, tke, taq, tqt, ttt, twt;
  if (!ws.loc.KendT || !encode_f32_blocks(&tw, ws.loc.W, units * C, D, D, C) ||
      !encode_f32_blocks(&tu, ws.loc.U, units * C, D, D, C) ||
      !encode_f32_blocks(&tkt, ws.loc.KendT, units * D, C, C, D) ||
      !encode_f32_blocks(&tke, ws.loc.Kend, units * C, D, D, C) ||
      !encode_f32_blocks(&taq, ws.loc.AqkT, units * C, C, C, C) ||
      !encode_f32_blocks(&tqt, ws.loc.QtT, units * D, C, C, D) ||
      !encode_f32_blocks(&ttt, ws.loc.TT, units * C, C, C, C) ||
      !encode_f32_blocks(&twt, ws.loc.WT, units * D, C, C, D))
    return cudaErrorNotSupported;
  const unsigned grid = seq_head_tile_ctas(P, D / BV);
  if (grid == 0) return cudaErrorInvalidConfiguration;
  auto fk = sbf16 ? bwd_fwd_scan_tc_kernel<true> : bwd_fwd_scan_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(fk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(F_DATA + 1024));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_rev_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(R_DATA + 1024));
  if (e != cudaSuccess) return e;
  fk<<<grid, NT, F_DATA + 1024, st>>>(P, ws, tw, tu, tkt, win, record ? 1 : 0);
  if ((e = cudaGetLastError()) != cudaSuccess || !record) return e;
  bwd_rev_scan_tc_kernel<<<grid, NT, R_DATA + 1024, st>>>(P, ws, A, tke, taq, tqt, ttt, twt, win);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------- pairwise terms
//
// Scalar decay: the pairwise decay exp(G_i - G_m) folds into dM and dA once per chunk
// (dM', dA'), and the three products the chain rule needs through A_qk = (Q^ K^T) o X and
// A_kk = diag(beta) (K^ K^T) o X are plain contractions over the chunk's tokens:
//
//   [dM'; dA'] K^           rows 0-63: P1 = dM' K^,  rows 64-127: P2 = dA' K^
//   [dM'^T | (b dA')^T] [Q^; K^]   P3 = dM'^T Q^ + (diag(beta) dA')^T K^
//
// on tensor cores (kind::tf32, K-major operands written by the threads: dM' and dA' as
// stored and transposed, Q^ and K^ transposed), staged to shared memory, then the same
// elementwise chain rule as bwd_pair_kernel: dq^, dk^, the rows of dG (whose reverse
// cumulative sum is dg), dbeta's pairwise part, and after the value heads of the key head
// the L2 normalisation's backward.

namespace bpt {

constexpr int C = 64, D = 128, NT = 512, DP = D + 4;
constexpr uint32_t Q_OFF = 0, K_OFF = C * DP * 4;                  // q^, k^ rows, fp32
constexpr uint32_t OPS = 2 * C * DP * 4;                           // 67584, 1024-aligned
constexpr uint32_t A12 = OPS;                                      // 2 blocks of 128 rows
constexpr uint32_t A3 = A12 + 32768;                               // 4 blocks of 64 rows
constexpr uint32_t BQ = A3 + 40960;                                // Q^T 2 blocks, then K^T 2
constexpr uint32_t BK = BQ + 32768;
constexpr uint32_t DATA = BK + 32768;                              // 206848
constexpr uint32_t SMALL = DATA;                                   // per-token and per-channel
constexpr uint32_t SMEM = DATA + 4096 + 1024;
constexpr int SP = DP;                                             // staging rows of P1-P3
constexpr uint32_t kWaitLimit = 1u << 22;
static_assert(3 * C * SP * 4 <= DATA - OPS, "P1-P3 staging fits the operand region");
static_assert(SMEM <= 227 * 1024, "shared memory budget");
static_assert(OPS % 1024 == 0, "operand alignment");

struct Ctrl {
  uint64_t bar;
  uint32_t tmem;
  int bad;
};

}  // namespace bpt

__global__ void __launch_bounds__(bpt::NT, 1)
    bwd_pair_tc_kernel(Problem P, BwdWorkspace ws, BwdArgs A, ChunkWindow win) {
  using namespace bpt;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* const data = smem_raw + pad;
  float* const s_q = reinterpret_cast<float*>(data + Q_OFF);
  float* const s_k = reinterpret_cast<float*>(data + K_OFF);
  float* const s_G = reinterpret_cast<float*>(data + SMALL);       // [C] cumulative log-decay
  float* const s_b = s_G + C;                                      // [C] beta
  float* const s_rq = s_b + C;                                     // [C] 1/|q|
  float* const s_rk = s_rq + C;                                    // [C] 1/|k|
  float* const s_db = s_rk + C;                                    // [C] dbeta's pairwise part
  float* const s_dot = s_db + C;                                   // [C] row sums of dG
  float* const s_dGl = s_dot + C;                                  // [D] gradient w.r.t. G_last
  Ctrl* const ctl = reinterpret_cast<Ctrl*>(s_dGl + D);
  constexpr int IR = C * 16 / NT, JC = D / 16;   // a thread's rows and columns of C x D tiles

  int gc;
  if (ws.loc.plan.info[1] == 0 || !window_chunk(ws.loc.plan, P.num_seqs, win, blockIdx.x, &gc)) return;
  const ChunkInfo ci = ws.loc.plan.chunks[gc];
  const int kh = blockIdx.y, HV = P.HV, ratio = HV / P.HK, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool delta = !(P.flags & KDA_FLAG_NO_DELTA);
  const int n = ci.n;
  const int r0 = (tid / 16) * IR, c0 = (tid % 16) * JC;
  const bool lead = (tid % 16) == 0;
  const uint32_t sd = tc::smem_u32(data);

  if (tid == 0) {
    tc::mbar_init(&ctl->bar, 1);
    ctl->bad = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&ctl->tmem, 256);
    tc::tmem_relinquish();
  }
  for (int u = tid; u < C * (D / 8); u += NT) {    // q, k rows of the key head (bf16)
    const int i = u / (D / 8), c = (u % (D / 8)) * 8;
    float qx[8] = {}, kx[8] = {};
    if (i < n) {
      tc::bf16x8_load(reinterpret_cast<const unsigned char*>(
                          static_cast<const uint16_t*>(P.q) + (ci.t0 + i) * P.q_stride + static_cast<int64_t>(kh) * D + c), qx);
      tc::bf16x8_load(reinterpret_cast<const unsigned char*>(
                          static_cast<const uint16_t*>(P.k) + (ci.t0 + i) * P.k_stride + static_cast<int64_t>(kh) * D + c), kx);
    }
    *reinterpret_cast<float4*>(s_q + i * DP + c) = make_float4(qx[0], qx[1], qx[2], qx[3]);
    *reinterpret_cast<float4*>(s_q + i * DP + c + 4) = make_float4(qx[4], qx[5], qx[6], qx[7]);
    *reinterpret_cast<float4*>(s_k + i * DP + c) = make_float4(kx[0], kx[1], kx[2], kx[3]);
    *reinterpret_cast<float4*>(s_k + i * DP + c + 4) = make_float4(kx[4], kx[5], kx[6], kx[7]);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem;
  for (int i = warp; i < C; i += NT / 32) {
    float sq = 0.f, sk = 0.f;
    for (int c = lane; c < D; c += 32) {
      sq += s_q[i * DP + c] * s_q[i * DP + c];
      sk += s_k[i * DP + c] * s_k[i * DP + c];
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    if (lane == 0) {
      s_rq[i] = P.l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
      s_rk[i] = P.l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < C * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    s_q[i * DP + c] *= s_rq[i] * P.scale;
    s_k[i * DP + c] *= s_rk[i];
  }

  float adq[IR][JC], adk[IR][JC];
#pragma unroll
  for (int a = 0; a < IR; ++a)
#pragma unroll
    for (int b = 0; b < JC; ++b) adq[a][b] = adk[a][b] = 0.f;
  const uint32_t id = tc::idesc_f16(128, 128, tc::kTF32);

  for (int h = kh * ratio, it = 0; h < (kh + 1) * ratio; ++h, ++it) {
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * HV + h;
    __syncthreads();                            // the previous head's staging is read
    if (warp == 0) {                            // cumulative log-decay: two rows a lane, one scan
      const float a = 2 * lane < n ? P.g[(ci.t0 + 2 * lane) * HV + h] : 0.f;
      const float b = 2 * lane + 1 < n ? P.g[(ci.t0 + 2 * lane + 1) * HV + h] : 0.f;
      float inc = a + b;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
      }
      s_G[2 * lane] = inc - b;
      s_G[2 * lane + 1] = inc;
    }
    for (int i = tid; i < C; i += NT) s_b[i] = i < n ? P.beta[(ci.t0 + i) * HV + h] : 0.f;
    for (int c = tid; c < D; c += NT) s_dGl[c] = 0.f;
    // Q^T and K^T (key channel rows, token columns)
    for (int idx = tid; idx < C * D; idx += NT) {
      const int c = idx % D, m = idx / D;
      const uint32_t off = (m >> 5) * 16384 + tc::sw128_offset(c, (m & 31) >> 2) + (m & 3) * 4;
      *reinterpret_cast<float*>(data + BQ + off) = tf32_nearest(s_q[m * DP + c]);
      *reinterpret_cast<float*>(data + BK + off) = tf32_nearest(s_k[m * DP + c]);
    }
    __syncthreads();                            // G and beta are in
    // dM' and dA' (decay folded), as stored for [dM'; dA'] and transposed for P3
    for (int idx = tid; idx < C * C; idx += NT) {
      const int i = idx / C, m = idx % C;
      const float x = m <= i ? expf(s_G[i] - s_G[m]) : 0.f;
      const float dm = ws.dM[unit * C * C + idx] * x, da = ws.dA[unit * C * C + idx] * x;
      const uint32_t cm = (m & 31) >> 2, wm = (m & 3) * 4, ci2 = (i & 31) >> 2, wi = (i & 3) * 4;
      *reinterpret_cast<float*>(data + A12 + (m >> 5) * 16384 + tc::sw128_offset(i, cm) + wm) = tf32_nearest(dm);
      *reinterpret_cast<float*>(data + A12 + (m >> 5) * 16384 + tc::sw128_offset(C + i, cm) + wm) = tf32_nearest(da);
      *reinterpret_cast<float*>(data + A3 + (i >> 5) * 8192 + tc::sw128_offset(m, ci2) + wi) = tf32_nearest(dm);
      *reinterpret_cast<float*>(data + A3 + (2 + (i >> 5)) * 8192 + tc::sw128_offset(m, ci2) + wi) =
          tf32_nearest(delta ? s_b[i] * da : 0.f);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int j = 0; j < 2; ++j) {             // [dM'; dA'] K^: K = tokens m
        const uint64_t da = tc::smem_desc_sw128(sd + A12 + j * 16384, 1024);
        const uint64_t db = tc::smem_desc_sw128(sd + BK + j * 16384, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_ss_tf32(tmem, tc::desc_add(da, 32 * k), tc::desc_add(db, 32 * k), id, (j | k) ? 1u : 0u);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {             // [dM'^T | (b dA')^T] [Q^; K^]: K = 2 x tokens
        const uint64_t da = tc::smem_desc_sw128(sd + A3 + j * 8192, 1024);
        const uint64_t db = tc::smem_desc_sw128(sd + BQ + j * 16384, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_ss_tf32(tmem + 128, tc::desc_add(da, 32 * k), tc::desc_add(db, 32 * k), id, (j | k) ? 1u : 0u);
      }
      tc::mma_commit(&ctl->bar);
    }
    // the contractions' rows of this thread, requested while the products run
    float gq[IR][JC], gk[IR][JC], ge[IR][JC];
#pragma unroll
    for (int a = 0; a < IR; ++a) {
      ld_row(gq[a], ws.dQt + unit * C * D + (r0 + a) * D + c0);
      ld_row(gk[a], ws.dKt + unit * C * D + (r0 + a) * D + c0);
      ld_row(ge[a], ws.dKe + unit * C * D + (r0 + a) * D + c0);
    }
    if (!tc::mbar_wait_bounded(&ctl->bar, static_cast<uint32_t>(it) & 1u, kWaitLimit)) ctl->bad = 1;
    tc::fence_after_sync();
    // stage P1, P2, P3 as rows of SP floats over the operands
    float* const s_P1 = reinterpret_cast<float*>(data + OPS);
    float* const s_P2 = s_P1 + C * SP;
    float* const s_P3 = s_P2 + C * SP;
    __syncthreads();                            // the operands are read by the MMAs only
    {
      const int qd = warp & 3, ch = warp >> 2;
      const int row = 32 * qd + lane;
      const uint32_t la = static_cast<uint32_t>(32 * qd) << 16;
      float* dst12 = row < C ? s_P1 + row * SP : s_P2 + (row - C) * SP;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {          // warp w: columns 32 (w / 4) ..
        uint32_t v[16];
        tc::tmem_ld16(tmem + la + 32 * ch + 16 * jj, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(dst12 + 32 * ch + 16 * jj + e) =
              make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
      }
      if (qd < 2) {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          uint32_t v[16];
          tc::tmem_ld16(tmem + la + 128 + 32 * ch + 16 * jj, v);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(s_P3 + row * SP + 32 * ch + 16 * jj + e) =
                make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    {
      const float Gl = s_G[C - 1], gam = expf(Gl);
      float gl[JC];
#pragma unroll
      for (int b = 0; b < JC; ++b) gl[b] = 0.f;
#pragma unroll
      for (int a = 0; a < IR; ++a) {
        const int i = r0 + a;
        float p1[JC], p2[JC], p3[JC], qv[JC], kv[JC];
        const float* dqt = gq[a];
        const float* dkt = gk[a];
        const float* dke = ge[a];
        ld_row(p1, s_P1 + i * SP + c0);
        ld_row(p2, s_P2 + i * SP + c0);
        ld_row(p3, s_P3 + i * SP + c0);
        ld_row(qv, s_q + i * DP + c0);
        ld_row(kv, s_k + i * DP + c0);
        const float bi = s_b[i], Gi = s_G[i];
        const float eG = expf(Gi), eL = expf(Gl - Gi);
        float bl = 0.f, rsum = 0.f;
#pragma unroll
        for (int b = 0; b < JC; ++b) {
          adq[a][b] += p1[b] + dqt[b] * eG;
          adk[a][b] += bi * p2[b] + p3[b] + dkt[b] * eG + dke[b] * eL;
          rsum += qv[b] * p1[b] + kv[b] * bi * p2[b] - kv[b] * p3[b] + dqt[b] * qv[b] * eG +
                  dkt[b] * kv[b] * eG - dke[b] * kv[b] * eL;
          bl += kv[b] * p2[b];                  // dbeta's pairwise part: sum_c k^_ic P2_ic
          gl[b] += dke[b] * kv[b] * eL;         // K_end's path into G_last
        }
        bl = halfwarp_sum(bl);
        rsum = halfwarp_sum(rsum);
        if (lead) {
          s_db[i] = bl;
          s_dot[i] = rsum;
        }
      }
#pragma unroll
      for (int b = 0; b < JC; ++b) atomicAdd(&s_dGl[c0 + b], gl[b]);
      __syncthreads();
      if (warp == 0) {                          // G_last's terms join the last row
        float v = 0.f;
        for (int c = lane; c < D; c += 32) v += s_dGl[c] + ws.dgam[unit * D + c] * gam;
        v = warp_sum(v);
        if (lane == 0) s_dot[C - 1] += v;
      }
      __syncthreads();
      if (warp == 0) {                          // dg = reverse cumulative sum of the rows
        const int i1 = C - 1 - 2 * lane, i0 = i1 - 1;    // lane l: rows 63 - 2l and 62 - 2l
        const float a = s_dot[i1], b = s_dot[i0];
        float inc = a + b;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, inc, off);
          if (lane >= off) inc += y;
        }
        if (i1 < n) A.dg[(ci.t0 + i1) * HV + h] = inc - b;
        if (i0 < n) A.dg[(ci.t0 + i0) * HV + h] = inc;
      }
      for (int i = tid; i < n; i += NT)
        A.dbeta[(ci.t0 + i) * HV + h] = ws.dbr[unit * C + i] + (delta ? s_db[i] : 0.f);
    }
  }
  // the L2 normalisation's backward: with u = x / |x|, dx = (du - u (u . du)) / |x|
  const float inv_s = 1.f / P.scale;
#pragma unroll
  for (int a = 0; a < IR; ++a) {
    const int i = r0 + a;
    float dq = 0.f, dk = 0.f;
#pragma unroll
    for (int b = 0; b < JC; ++b) {
      dq += s_q[i * DP + c0 + b] * adq[a][b];
      dk += s_k[i * DP + c0 + b] * adk[a][b];
    }
    dq = halfwarp_sum(dq);
    dk = halfwarp_sum(dk);
    if (i >= n) continue;
    float oq[JC], ok[JC];
#pragma unroll
    for (int b = 0; b < JC; ++b) {
      if (P.l2norm) {
        const float uq = s_q[i * DP + c0 + b] * inv_s;
        oq[b] = P.scale * s_rq[i] * (adq[a][b] - uq * dq * inv_s);
        ok[b] = s_rk[i] * (adk[a][b] - s_k[i * DP + c0 + b] * dk);
      } else {
        oq[b] = P.scale * adq[a][b];
        ok[b] = adk[a][b];
      }
    }
    const int64_t o = ((ci.t0 + i) * P.HK + kh) * D + c0;
    st_row(A.dq + o, oq);
    st_row(A.dk + o, ok);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (ctl->bad && tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// Per-channel decay: with the anchor G_a at the chunk's middle token and E+ = exp(G - G_a), the
// pairwise factor exp(G_ic - G_mc) is E+_ic / E+_mc, so the three products take anchored
// operands and are rescaled after:
//
//   [dM; dA] K-^T          P1 = E+ o (dM K-),  P2 = E+ o (dA K-),   K- = k^ / E+
//   [dM^T | (b dA)^T] [(q^ E+); (k^ E+)]     P3 = (...) / E+
//
// (bwd_pair_kernel's anchored branch, on tensor cores).  A chunk whose decay leaves the anchor's
// range (80 nats) for some value head of the group is left to bwd_pair_kernel: the CTA records
// it in ws.pair_fb and writes no dq or dk.

namespace bpc {

constexpr int C = 64, D = 128, NT = 512, DP = D + 4, SP = DP;
constexpr uint32_t S_Q = 0, S_K = C * DP * 4, S_G = 2 * C * DP * 4;
constexpr uint32_t OPS = 3 * C * DP * 4;                           // 101376, 1024-aligned
// first products: [dM; dA] (2 blocks of 128 rows) and K-^T (2 blocks of 128 rows); second:
// [dM^T | (b dA)^T] (4 blocks of 64 rows + 8 KB under the last M = 128 read) and
// [(q^ E+)^T; (k^ E+)^T] (4 blocks of 128 rows); then the staged P1, P2, P3
constexpr uint32_t A12 = OPS, B12 = OPS + 32768;
constexpr uint32_t A3 = OPS, B3 = OPS + 40960;
constexpr uint32_t DATA = OPS + 40960 + 65536;                    // 207872
constexpr uint32_t SMALL = DATA;
constexpr uint32_t SMEM = DATA + 4096 + 1024;
constexpr uint32_t kWaitLimit = 1u << 22;
static_assert(OPS % 1024 == 0, "operand alignment");
static_assert(3 * C * SP * 4 <= DATA - OPS, "P1-P3 staging fits the operand region");
static_assert(SMEM <= 227 * 1024, "shared memory budget");

struct Ctrl {
  uint64_t bar;
  uint32_t tmem;
  int bad;
  int fb;                                                          // a head left the anchor's range
};

}  // namespace bpc

__global__ void __launch_bounds__(bpc::NT, 1)
    bwd_pair_tc_pc_kernel(Problem P, BwdWorkspace ws, BwdArgs A, ChunkWindow win) {
  using namespace bpc;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* const data = smem_raw + pad;
  float* const s_q = reinterpret_cast<float*>(data + S_Q);
  float* const s_k = reinterpret_cast<float*>(data + S_K);
  float* const s_G = reinterpret_cast<float*>(data + S_G);        // [C][DP] cumulative log-decay
  float* const s_b = reinterpret_cast<float*>(data + SMALL);       // [C] beta
  float* const s_rq = s_b + C;                                     // [C] 1/|q|
  float* const s_rk = s_rq + C;                                    // [C] 1/|k|
  float* const s_db = s_rk + C;                                    // [C] dbeta's pairwise part
  float* const s_ga = s_db + C;                                    // [D] G at the anchor token
  float* const s_dGl = s_ga + D;                                   // [D] gradient w.r.t. G_last
  float* const s_gam = s_dGl + D;                                  // [D] exp(G_last)
  Ctrl* const ctl = reinterpret_cast<Ctrl*>(s_gam + D);
  constexpr int IR = C * 16 / NT, JC = D / 16;

  int gc;
  if (ws.loc.plan.info[1] == 0 || !window_chunk(ws.loc.plan, P.num_seqs, win, blockIdx.x, &gc)) return;
  const ChunkInfo ci = ws.loc.plan.chunks[gc];
  const int kh = blockIdx.y, HV = P.HV, ratio = HV / P.HK, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool delta = !(P.flags & KDA_FLAG_NO_DELTA);
  const int n = ci.n;
  const int r0 = (tid / 16) * IR, c0 = (tid % 16) * JC;
  const bool lead = (tid % 16) == 0;
  const uint32_t sd = tc::smem_u32(data);

  if (tid == 0) {
    tc::mbar_init(&ctl->bar, 1);
    ctl->bad = 0;
    ctl->fb = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&ctl->tmem, 256);
    tc::tmem_relinquish();
  }
  for (int u = tid; u < C * (D / 8); u += NT) {    // q, k rows of the key head (bf16)
    const int i = u / (D / 8), c = (u % (D / 8)) * 8;
    float qx[8] = {}, kx[8] = {};
    if (i < n) {
      tc::bf16x8_load(reinterpret_cast<const unsigned char*>(
                          static_cast<const uint16_t*>(P.q) + (ci.t0 + i) * P.q_stride + static_cast<int64_t>(kh) * D + c), qx);
      tc::bf16x8_load(reinterpret_cast<const unsigned char*>(
                          static_cast<const uint16_t*>(P.k) + (ci.t0 + i) * P.k_stride + static_cast<int64_t>(kh) * D + c), kx);
    }
    st_row(s_q + i * DP + c, qx);
    st_row(s_k + i * DP + c, kx);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem;
  for (int i = warp; i < C; i += NT / 32) {
    float sq = 0.f, sk = 0.f;
    for (int c = lane; c < D; c += 32) {
      sq += s_q[i * DP + c] * s_q[i * DP + c];
      sk += s_k[i * DP + c] * s_k[i * DP + c];
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    if (lane == 0) {
      s_rq[i] = P.l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
      s_rk[i] = P.l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < C * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    s_q[i * DP + c] *= s_rq[i] * P.scale;
    s_k[i * DP + c] *= s_rk[i];
  }

  float adq[IR][JC], adk[IR][JC];
#pragma unroll
  for (int a = 0; a < IR; ++a)
#pragma unroll
    for (int b = 0; b < JC; ++b) adq[a][b] = adk[a][b] = 0.f;
  const uint32_t id = tc::idesc_f16(128, 128, tc::kTF32);
  uint32_t phase = 0;
  const int am = (n - 1) / 2;                   // the anchor token

  for (int h = kh * ratio; h < (kh + 1) * ratio; ++h) {
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * HV + h;
    __syncthreads();                            // the previous head's staging is read
    for (int idx = tid; idx < C * D; idx += NT) {
      const int i = idx / D, c = idx % D;
      s_G[i * DP + c] = i < n ? P.g[((ci.t0 + i) * HV + h) * D + c] : 0.f;
    }
    for (int i = tid; i < C; i += NT) s_b[i] = i < n ? P.beta[(ci.t0 + i) * HV + h] : 0.f;
    for (int c = tid; c < D; c += NT) s_dGl[c] = 0.f;
    __syncthreads();
    if (tid < D) {                              // cumulative log-decay down each channel
      float acc = 0.f;
      for (int i = 0; i < C; ++i) {
        acc += s_G[i * DP + tid];
        s_G[i * DP + tid] = acc;
      }
      s_ga[tid] = s_G[am * DP + tid];
      s_gam[tid] = expf(acc);
    }
    __syncthreads();
    bool wide = false;
    for (int idx = tid; idx < C * D; idx += NT) {
      const int i = idx / D, c = idx % D;
      wide |= fabsf(s_G[i * DP + c] - s_ga[c]) > kSimtAnchorRange;
    }
    if (__syncthreads_or(wide)) {               // left to the exact CUDA-core kernel
      if (tid == 0) ctl->fb = 1;
      continue;
    }
    // [dM; dA] as stored and K-^T (key channel rows, token columns)
    for (int idx = tid; idx < C * C; idx += NT) {
      const int i = idx / C, m = idx % C;
      const uint32_t cm = (m & 31) >> 2, wm = (m & 3) * 4;
      *reinterpret_cast<float*>(data + A12 + (m >> 5) * 16384 + tc::sw128_offset(i, cm) + wm) =
          tf32_nearest(ws.dM[unit * C * C + idx]);
      *reinterpret_cast<float*>(data + A12 + (m >> 5) * 16384 + tc::sw128_offset(C + i, cm) + wm) =
          tf32_nearest(ws.dA[unit * C * C + idx]);
    }
    for (int idx = tid; idx < C * D; idx += NT) {
      const int m = idx / D, c = idx % D;
      const float km = s_k[m * DP + c] * expf(s_ga[c] - s_G[m * DP + c]);
      *reinterpret_cast<float*>(data + B12 + (m >> 5) * 16384 + tc::sw128_offset(c, (m & 31) >> 2) + (m & 3) * 4) =
          tf32_nearest(km);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint64_t da = tc::smem_desc_sw128(sd + A12 + j * 16384, 1024);
        const uint64_t db = tc::smem_desc_sw128(sd + B12 + j * 16384, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_ss_tf32(tmem, tc::desc_add(da, 32 * k), tc::desc_add(db, 32 * k), id, (j | k) ? 1u : 0u);
      }
      tc::mma_commit(&ctl->bar);
    }
    if (!tc::mbar_wait_bounded(&ctl->bar, phase & 1u, kWaitLimit)) ctl->bad = 1;
    ++phase;
    tc::fence_after_sync();
    __syncthreads();                            // the first operands are read
    // [dM^T | (b dA)^T] and [(q^ E+)^T; (k^ E+)^T]
    for (int idx = tid; idx < C * C; idx += NT) {
      const int i = idx / C, m = idx % C;
      const uint32_t ci2 = (i & 31) >> 2, wi = (i & 3) * 4;
      *reinterpret_cast<float*>(data + A3 + (i >> 5) * 8192 + tc::sw128_offset(m, ci2) + wi) =
          tf32_nearest(ws.dM[unit * C * C + idx]);
      *reinterpret_cast<float*>(data + A3 + (2 + (i >> 5)) * 8192 + tc::sw128_offset(m, ci2) + wi) =
          tf32_nearest(delta ? s_b[i] * ws.dA[unit * C * C + idx] : 0.f);
    }
    for (int idx = tid; idx < C * D; idx += NT) {
      const int m = idx / D, c = idx % D;
      const float e = expf(s_G[m * DP + c] - s_ga[c]);
      const uint32_t off = (m >> 5) * 16384 + tc::sw128_offset(c, (m & 31) >> 2) + (m & 3) * 4;
      *reinterpret_cast<float*>(data + B3 + off) = tf32_nearest(s_q[m * DP + c] * e);
      *reinterpret_cast<float*>(data + B3 + 32768 + off) = tf32_nearest(s_k[m * DP + c] * e);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t da = tc::smem_desc_sw128(sd + A3 + j * 8192, 1024);
        const uint64_t db = tc::smem_desc_sw128(sd + B3 + j * 16384, 1024);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_ss_tf32(tmem + 128, tc::desc_add(da, 32 * k), tc::desc_add(db, 32 * k), id, (j | k) ? 1u : 0u);
      }
      tc::mma_commit(&ctl->bar);
    }
    // the contractions' rows of this thread, requested while the second products run
    float gq[IR][JC], gk[IR][JC], ge[IR][JC];
#pragma unroll
    for (int a = 0; a < IR; ++a) {
      ld_row(gq[a], ws.dQt + unit * C * D + (r0 + a) * D + c0);
      ld_row(gk[a], ws.dKt + unit * C * D + (r0 + a) * D + c0);
      ld_row(ge[a], ws.dKe + unit * C * D + (r0 + a) * D + c0);
    }
    if (!tc::mbar_wait_bounded(&ctl->bar, phase & 1u, kWaitLimit)) ctl->bad = 1;
    ++phase;
    tc::fence_after_sync();
    float* const s_P1 = reinterpret_cast<float*>(data + OPS);
    float* const s_P2 = s_P1 + C * SP;
    float* const s_P3 = s_P2 + C * SP;
    __syncthreads();                            // the second operands are read
    {
      const int qd = warp & 3, ch = warp >> 2;
      const int row = 32 * qd + lane;
      const uint32_t la = static_cast<uint32_t>(32 * qd) << 16;
      float* dst12 = row < C ? s_P1 + row * SP : s_P2 + (row - C) * SP;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        uint32_t v[16];
        tc::tmem_ld16(tmem + la + 32 * ch + 16 * jj, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(dst12 + 32 * ch + 16 * jj + e) =
              make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
      }
      if (qd < 2) {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          uint32_t v[16];
          tc::tmem_ld16(tmem + la + 128 + 32 * ch + 16 * jj, v);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(s_P3 + row * SP + 32 * ch + 16 * jj + e) =
                make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    {
      // the rescaled products and the chain rule; dG_ic in place of P1_ic
      float gl[JC];
#pragma unroll
      for (int b = 0; b < JC; ++b) gl[b] = 0.f;
#pragma unroll
      for (int a = 0; a < IR; ++a) {
        const int i = r0 + a;
        float p1[JC], p2[JC], p3[JC], qv[JC], kv[JC], gi[JC], ga[JC], glast[JC];
        ld_row(p1, s_P1 + i * SP + c0);
        ld_row(p2, s_P2 + i * SP + c0);
        ld_row(p3, s_P3 + i * SP + c0);
        ld_row(qv, s_q + i * DP + c0);
        ld_row(kv, s_k + i * DP + c0);
        ld_row(gi, s_G + i * DP + c0);
        ld_row(ga, s_ga + c0);
        ld_row(glast, s_G + (C - 1) * DP + c0);
        const float bi = s_b[i];
        float bl = 0.f, dgr[JC];
#pragma unroll
        for (int b = 0; b < JC; ++b) {
          const float d = gi[b] - ga[b];
          const float ep = expf(d), em = expf(-d);
          const float eG = expf(gi[b]), eL = expf(glast[b] - gi[b]);
          const float q1 = p1[b] * ep, q2 = p2[b] * ep, q3 = p3[b] * em;
          const float dqt = gq[a][b], dkt = gk[a][b], dke = ge[a][b];
          adq[a][b] += q1 + dqt * eG;
          adk[a][b] += bi * q2 + q3 + dkt * eG + dke * eL;
          dgr[b] = qv[b] * q1 + kv[b] * bi * q2 - kv[b] * q3 + dqt * qv[b] * eG + dkt * kv[b] * eG -
                   dke * kv[b] * eL;
          bl += kv[b] * q2;                     // dbeta's pairwise part: sum_c k^_ic P2_ic
          gl[b] += dke * kv[b] * eL;            // K_end's path into G_last
        }
        st_row(s_P1 + i * SP + c0, dgr);
        bl = halfwarp_sum(bl);
        if (lead) s_db[i] = bl;
      }
#pragma unroll
      for (int b = 0; b < JC; ++b) atomicAdd(&s_dGl[c0 + b], gl[b]);
      __syncthreads();
      if (tid < D) {                            // dg = reverse cumulative sum down each channel
        float acc = s_dGl[tid] + ws.dgam[unit * D + tid] * s_gam[tid];
        for (int i = C - 1; i >= 0; --i) {
          acc += s_P1[i * SP + tid];
          if (i < n) A.dg[((ci.t0 + i) * HV + h) * D + tid] = acc;
        }
      }
      for (int i = tid; i < n; i += NT)
        A.dbeta[(ci.t0 + i) * HV + h] = ws.dbr[unit * C + i] + (delta ? s_db[i] : 0.f);
    }
  }
  // a head outside the anchor's range: bwd_pair_kernel redoes the whole chunk and key head
  __syncthreads();
  const bool fb = ctl->fb != 0;
  if (tid == 0) ws.pair_fb[static_cast<int64_t>(blockIdx.x) * P.HK + kh] = fb ? 1 : 0;
  if (!fb) {
    const float inv_s = 1.f / P.scale;
#pragma unroll
    for (int a = 0; a < IR; ++a) {
      const int i = r0 + a;
      float dq = 0.f, dk = 0.f;
#pragma unroll
      for (int b = 0; b < JC; ++b) {
        dq += s_q[i * DP + c0 + b] * adq[a][b];
        dk += s_k[i * DP + c0 + b] * adk[a][b];
      }
      dq = halfwarp_sum(dq);
      dk = halfwarp_sum(dk);
      if (i >= n) continue;
      float oq[JC], ok[JC];
#pragma unroll
      for (int b = 0; b < JC; ++b) {
        if (P.l2norm) {
          const float uq = s_q[i * DP + c0 + b] * inv_s;
          oq[b] = P.scale * s_rq[i] * (adq[a][b] - uq * dq * inv_s);
          ok[b] = s_rk[i] * (adk[a][b] - s_k[i * DP + c0 + b] * dk);
        } else {
          oq[b] = P.scale * adq[a][b];
          ok[b] = adk[a][b];
        }
      }
      const int64_t o = ((ci.t0 + i) * P.HK + kh) * D + c0;
      st_row(A.dq + o, oq);
      st_row(A.dk + o, ok);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (ctl->bad && tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

cudaError_t launch_bwd_pair_tc(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A, ChunkWindow win,
                               int slots, bool perch, cudaStream_t st) {
  using namespace bpt;
  if (slots <= 0) return cudaSuccess;
  if (perch) {
    cudaError_t e = cudaFuncSetAttribute(bwd_pair_tc_pc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bpc::SMEM));
    if (e != cudaSuccess) return e;
    bwd_pair_tc_pc_kernel<<<dim3(static_cast<unsigned>(slots), P.HK), bpc::NT, bpc::SMEM, st>>>(P, ws, A, win);
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(bwd_pair_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM));
  if (e != cudaSuccess) return e;
  bwd_pair_tc_kernel<<<dim3(static_cast<unsigned>(slots), P.HK), NT, SMEM, st>>>(P, ws, A, win);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------- local stage
//
// The chunk-local stage for scalar decay with its products on tensor cores (kind::tf32):
//
//   [K^; Q^] K^T      rows 0-63: K^ K^T, rows 64-127: Q^ K^T   (then the decay, beta and the
//                     masks on the CUDA cores: A_kk, A_qk)
//   T = (I + A_kk)^-1 on the CUDA cores (tri_unit_lower_inverse)
//   (beta K~)^T T^T = W^T,  (beta V)^T T^T = U^T        (M = 128 key channels / value columns)
//
// and the element-wise rest (K~, Q~, K_end, gamma), writing the same workspace arrays as
// simt_local_kernel does for the tensor-core scans, the MMA operands among them rounded to tf32.

namespace blt {

constexpr int C = 64, D = 128, NT = 512, DP = D + 4, CP = C + 4;
constexpr int CW = 64 / (NT / 128);             // accumulator columns a warp reads (16)
constexpr uint32_t S_K = 0, S_V = C * DP * 4;                       // k^, v rows (fp32)
constexpr uint32_t OPS = 2 * C * DP * 4;                            // 67584, 1024-aligned
// first products: [K^; Q^] as 4 blocks of 128 rows (K = key channels); the second: (beta K~)^T
// and (beta V)^T as 2 blocks of 128 rows each (K = tokens), T as 2 blocks of 64 rows
constexpr uint32_t A_W = OPS, A_U = OPS + 32768, B_T = OPS + 65536;
constexpr uint32_t S_A = OPS + 81920, S_AQ = S_A + C * CP * 4, S_T = S_AQ + C * CP * 4,
                   S_X = S_T + C * CP * 4, SMALL = S_X + C * CP * 4;
constexpr uint32_t SMEM = SMALL + 3072 + 64 + 1024;                // small arrays, control, slack
constexpr uint32_t kWaitLimit = 1u << 22;
static_assert(C * DP * 4 <= 2 * C * CP * 4, "q rows fit over T and X");
static_assert((6 * C + 3 * D) * 4 + 16 <= 3072 + 64, "small arrays and the control block");
static_assert(4 * 8192 <= 2 * C * CP * 4 && S_A % 1024 == 0, "K- operand over A_kk and A_qk");
static_assert(SMEM <= 227 * 1024, "shared memory budget");

struct Ctrl {
  uint64_t bar;
  uint32_t tmem;
  int bad;
};

}  // namespace blt

// PERCH: per-channel decay with factors anchored at the chunk's middle token, K+ = k^ E+,
// Q+ = q^ E+, K- = k^ / E+ (E+ = exp(G - G_a)): [K+; Q+] K-^T carries the pairwise decay
// exp(G_ic - G_jc) inside the product (simt_local_kernel's anchored branch).  A chunk whose decay
// leaves the anchor's range (80 nats) is flagged in ws.local_fb and left to simt_local_kernel.
template <bool PERCH>
__global__ void __launch_bounds__(blt::NT, 1)
    bwd_local_tc_kernel(Problem P, SimtWorkspace ws, ChunkWindow win) {
  using namespace blt;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t pad = (1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char* const data = smem_raw + pad;
  float* const s_k = reinterpret_cast<float*>(data + S_K);
  float* const s_v = reinterpret_cast<float*>(data + S_V);          // scalar: v rows
  float* const s_Gc = reinterpret_cast<float*>(data + S_V);         // per channel: G, then K-
  float* const s_q = reinterpret_cast<float*>(data + S_T);          // until A_qk is formed
  float* const s_A = reinterpret_cast<float*>(data + S_A);
  float* const s_Aq = reinterpret_cast<float*>(data + S_AQ);
  float* const s_T = reinterpret_cast<float*>(data + S_T);
  float* const s_X = reinterpret_cast<float*>(data + S_X);
  float* const s_G = reinterpret_cast<float*>(data + SMALL);       // [C]
  float* const s_beta = s_G + C;                                   // [C]
  float* const s_inv = s_beta + C;                                 // [2C]
  float* const s_eG = s_inv + 2 * C;                               // [C] exp(G_i)
  float* const s_eL = s_eG + C;                                    // [C] exp(G_last - G_i)
  float* const s_ga = s_eL + C;                                    // [D] per channel: G_a
  float* const s_eA = s_ga + D;                                    // [D] exp(G_a)
  float* const s_eLA = s_eA + D;                                   // [D] exp(G_last - G_a)
  Ctrl* const ctl = reinterpret_cast<Ctrl*>(s_eLA + D);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int gc;
  if (ws.plan.info[1] == 0 || !window_chunk(ws.plan, P.num_seqs, win, blockIdx.x, &gc)) return;
  const ChunkInfo ci = ws.plan.chunks[gc];
  const int h = blockIdx.y, HV = P.HV, kh = h / (HV / P.HK), n = ci.n;
  const int64_t t0 = ci.t0;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * HV + h;
  const bool delta = !(P.flags & KDA_FLAG_NO_DELTA);
  const uint32_t sd = tc::smem_u32(data);

  if (tid == 0) {
    tc::mbar_init(&ctl->bar, 1);
    ctl->bad = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&ctl->tmem, 256);
    tc::tmem_relinquish();
  }
  for (int u = tid; u < C * (D / 8); u += NT) {    // k, q (key head), v or g (value head)
    const int i = u / (D / 8), c = (u % (D / 8)) * 8;
    float kx[8] = {}, qx[8] = {}, vx[8] = {};
    if (i < n) {
      const int64_t t = t0 + i;
      tc::bf16x8_load(reinterpret_cast<const unsigned char*>(static_cast<const uint16_t*>(P.k) + t * P.k_stride +
                                                              static_cast<int64_t>(kh) * D + c), kx);
      tc::bf16x8_load(reinterpret_cast<const unsigned char*>(static_cast<const uint16_t*>(P.q) + t * P.q_stride +
                                                              static_cast<int64_t>(kh) * D + c), qx);
      if constexpr (PERCH) {                    // log-decay: 4-byte aligned, so scalar loads
        const float* gp = P.g + (t * HV + h) * D + c;
#pragma unroll
        for (int e = 0; e < 8; ++e) vx[e] = gp[e];
      } else {
        tc::bf16x8_load(reinterpret_cast<const unsigned char*>(static_cast<const uint16_t*>(P.v) + t * P.v_stride +
                                                                static_cast<int64_t>(h) * D + c), vx);
      }
    }
    st_row(s_k + i * DP + c, kx);
    st_row(s_q + i * DP + c, qx);
    st_row(s_v + i * DP + c, vx);
  }
  for (int i = tid; i < C; i += NT) {
    const bool live = i < n;
    s_beta[i] = live ? P.beta[(t0 + i) * HV + h] : 0.f;
    if (!PERCH) s_G[i] = live ? P.g[(t0 + i) * HV + h] : 0.f;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem;
  for (int i = warp; i < C; i += NT / 32) {       // L2 norms and the query scale
    float sk = 0.f, sq = 0.f;
    for (int c = lane; c < D; c += 32) {
      sk += s_k[i * DP + c] * s_k[i * DP + c];
      sq += s_q[i * DP + c] * s_q[i * DP + c];
    }
    sk = warp_sum(sk);
    sq = warp_sum(sq);
    if (lane == 0) {
      s_inv[i] = P.l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
      s_inv[C + i] = (P.l2norm ? rsqrtf(sq + 1e-6f) : 1.f) * P.scale;
    }
  }
  if (!PERCH && warp == 0) {                    // inclusive cumulative log-decay, two rows a lane
    const float a = s_G[2 * lane], b = s_G[2 * lane + 1];
    float inc = a + b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    s_G[2 * lane] = inc - b;
    s_G[2 * lane + 1] = inc;
  }
  if (PERCH && tid < D) {                       // down each channel; the anchor's factors
    float acc = 0.f;
    for (int i = 0; i < C; ++i) {
      acc += s_Gc[i * DP + tid];
      s_Gc[i * DP + tid] = acc;
    }
    const float ga = s_Gc[((n - 1) / 2) * DP + tid];
    s_ga[tid] = ga;
    s_eA[tid] = expf(ga);
    s_eLA[tid] = expf(acc - ga);
    ws.gamma[unit * D + tid] = expf(acc);
  }
  __syncthreads();
  if constexpr (PERCH) {                        // out of the anchor's range: the exact kernel
    bool wide = false;
    for (int idx = tid; idx < C * D; idx += NT)
      wide |= fabsf(s_Gc[(idx / D) * DP + idx % D] - s_ga[idx % D]) > kSimtAnchorRange;
    wide = __syncthreads_or(wide);
    if (tid == 0) ws.local_fb[unit] = wide ? 1 : 0;
    if (wide) {
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (warp == 0) tc::tmem_dealloc(tmem, 256);
      return;
    }
  }
  // [K^; Q^] (per channel [K+; Q+]) rows into the first operand, float4 pieces of 4 key
  // channels; per channel also K- into the second operand over A_kk and A_qk
  const float Gl = s_G[C - 1];
  if (!PERCH)
    for (int i = tid; i < C; i += NT) {
      s_eG[i] = expf(s_G[i]);
      s_eL[i] = expf(Gl - s_G[i]);
    }
  for (int u = tid; u < C * (D / 4); u += NT) {
    const int i = u / (D / 4), c = (u % (D / 4)) * 4;
    float4 k4 = *reinterpret_cast<float4*>(s_k + i * DP + c);
    float4 q4 = *reinterpret_cast<float4*>(s_q + i * DP + c);
    const float sk = s_inv[i], sq = s_inv[C + i];
    float kx[4] = {k4.x * sk, k4.y * sk, k4.z * sk, k4.w * sk};
    float qx[4] = {q4.x * sq, q4.y * sq, q4.z * sq, q4.w * sq};
    if constexpr (PERCH) {
      float km[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float d = s_Gc[i * DP + c + e] - s_ga[c + e];
        const float ep = expf(d), em = expf(-d);
        km[e] = kx[e] * em;
        kx[e] *= ep;
        qx[e] *= ep;
      }
      *reinterpret_cast<float4*>(s_Gc + i * DP + c) = make_float4(km[0], km[1], km[2], km[3]);
      *reinterpret_cast<float4*>(data + S_A + (c >> 5) * 8192 + tc::sw128_offset(i, (c & 31) >> 2)) =
          make_float4(tf32_nearest(km[0]), tf32_nearest(km[1]), tf32_nearest(km[2]), tf32_nearest(km[3]));
    }
    *reinterpret_cast<float4*>(s_k + i * DP + c) = make_float4(kx[0], kx[1], kx[2], kx[3]);
    *reinterpret_cast<float4*>(s_q + i * DP + c) = make_float4(qx[0], qx[1], qx[2], qx[3]);
    *reinterpret_cast<float4*>(data + OPS + (c >> 5) * 16384 + tc::sw128_offset(i, (c & 31) >> 2)) =
        make_float4(tf32_nearest(kx[0]), tf32_nearest(kx[1]), tf32_nearest(kx[2]), tf32_nearest(kx[3]));
    *reinterpret_cast<float4*>(data + OPS + (c >> 5) * 16384 + tc::sw128_offset(C + i, (c & 31) >> 2)) =
        make_float4(tf32_nearest(qx[0]), tf32_nearest(qx[1]), tf32_nearest(qx[2]), tf32_nearest(qx[3]));
  }
  if (!PERCH)
    for (int c = tid; c < D; c += NT) ws.gamma[unit * D + c] = expf(Gl);
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0) {                               // [K^; Q^] K^T (K^ the operand's rows 0-63), or [K+; Q+] K-^T
    tc::fence_after_sync();
    const uint32_t id = tc::idesc_f16(128, 64, tc::kTF32);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint64_t da = tc::smem_desc_sw128(sd + OPS + j * 16384, 1024);
      const uint64_t db = PERCH ? tc::smem_desc_sw128(sd + S_A + j * 8192, 1024) : da;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc::mma_ss_tf32(tmem, tc::desc_add(da, 32 * k), tc::desc_add(db, 32 * k), id, (j | k) ? 1u : 0u);
    }
    tc::mma_commit(&ctl->bar);
  }
  if (!tc::mbar_wait_bounded(&ctl->bar, 0, kWaitLimit)) ctl->bad = 1;
  tc::fence_after_sync();
  // A_kk and A_qk from the products: the decay exp(G_i - G_j) (scalar), beta and the masks
  const int qd = warp & 3, ch = warp >> 2;
  const int row = 32 * qd + lane;               // TMEM lane
  const uint32_t la = static_cast<uint32_t>(32 * qd) << 16;
  {
    uint32_t v0[16];
    tc::tmem_ld16(tmem + la + CW * ch, v0);
    tc::tmem_wait_ld();
    const int i = row & (C - 1);
    const float Gi = PERCH ? 0.f : s_G[i], bi = s_beta[i];
    float* dst = (row < C ? s_A : s_Aq) + i * CP + CW * ch;
#pragma unroll
    for (int e = 0; e < CW; ++e) {
      const int j = CW * ch + e;
      const float x = __uint_as_float(v0[e]);
      const float dec = j <= i ? (PERCH ? 1.f : expf(Gi - s_G[j])) : 0.f;
      dst[e] = row < C ? ((delta && j < i) ? bi * x * dec : 0.f) : x * dec;
    }
  }
  // the element-wise outputs of k^ and q^: K~ (fp32), K_end (tf32) as rows; K_end^T and Q~^T
  // (tf32) through a transposing stage over the first operand (free once its product is done),
  // rows of 65 floats so that neither side of the transpose meets bank conflicts
  float* const stg_kt = reinterpret_cast<float*>(data + OPS);
  float* const stg_qt = stg_kt + D * (C + 1);
  for (int idx = tid; idx < C * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    // K~ = k^ exp(G), K_end = k^ exp(G_last - G), Q~ = q^ exp(G); per channel from K+, K-, Q+
    const float kv = s_k[i * DP + c], qv = s_q[i * DP + c];
    const float eG = PERCH ? s_eA[c] : s_eG[i];
    const float ke = tf32_nearest(PERCH ? s_Gc[i * DP + c] * s_eLA[c] : kv * s_eL[i]);
    ws.Kt[(unit * C + i) * D + c] = kv * eG;
    ws.Kend[(unit * C + i) * D + c] = ke;
    stg_kt[c * (C + 1) + i] = ke;
    stg_qt[c * (C + 1) + i] = tf32_nearest(qv * eG);
  }
  tc::fence_before_sync();
  __syncthreads();                              // the q rows over T and X are dead
  for (int idx = tid; idx < C * D; idx += NT) {
    const int c = idx / C, i = idx % C;
    ws.KendT[(unit * D + c) * C + i] = stg_kt[c * (C + 1) + i];
    ws.QtT[(unit * D + c) * C + i] = stg_qt[c * (C + 1) + i];
  }
  for (int idx = tid; idx < C * CP; idx += NT) s_T[idx] = 0.f;
  __syncthreads();
  tri_unit_lower_inverse<C, CP, NT>(s_A, s_T, s_X, tid);
  // (beta K~)^T and (beta V)^T (rows: key channel / value column, K = token), T (rows i, K = j)
  for (int u = tid; u < 2 * D * (C / 4); u += NT) {
    const int which = u / (D * (C / 4)), rem = u % (D * (C / 4));
    const int c = rem % D, j0 = (rem / D) * 4;
    float x[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = j0 + e;
      float vj;
      if constexpr (PERCH)                      // the value rows straight from global memory
        vj = (which == 1 && j < n) ? bf16_bits_to_f32(static_cast<const uint16_t*>(P.v)[(t0 + j) * P.v_stride +
                                                                                     static_cast<int64_t>(h) * D + c])
                                   : 0.f;
      else
        vj = s_v[j * DP + c];
      x[e] = which == 0 ? (delta ? s_beta[j] * s_k[j * DP + c] * (PERCH ? s_eA[c] : s_eG[j]) : 0.f)
                        : s_beta[j] * vj;
    }
    *reinterpret_cast<float4*>(data + (which ? A_U : A_W) + (j0 >> 5) * 16384 + tc::sw128_offset(c, (j0 & 31) >> 2)) =
        make_float4(tf32_nearest(x[0]), tf32_nearest(x[1]), tf32_nearest(x[2]), tf32_nearest(x[3]));
  }
  for (int u = tid; u < C * (C / 4); u += NT) {
    const int i = u / (C / 4), j0 = (u % (C / 4)) * 4;
    const float4 t = *reinterpret_cast<const float4*>(s_T + i * CP + j0);
    *reinterpret_cast<float4*>(data + B_T + (j0 >> 5) * 8192 + tc::sw128_offset(i, (j0 & 31) >> 2)) =
        make_float4(tf32_nearest(t.x), tf32_nearest(t.y), tf32_nearest(t.z), tf32_nearest(t.w));
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    tc::fence_after_sync();
    const uint32_t id = tc::idesc_f16(128, 64, tc::kTF32);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint64_t dt = tc::smem_desc_sw128(sd + B_T + j * 8192, 1024);
      const uint64_t dw = tc::smem_desc_sw128(sd + A_W + j * 16384, 1024);
      const uint64_t du = tc::smem_desc_sw128(sd + A_U + j * 16384, 1024);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tc::mma_ss_tf32(tmem + 64, tc::desc_add(dw, 32 * k), tc::desc_add(dt, 32 * k), id, (j | k) ? 1u : 0u);
        tc::mma_ss_tf32(tmem + 128, tc::desc_add(du, 32 * k), tc::desc_add(dt, 32 * k), id, (j | k) ? 1u : 0u);
      }
    }
    tc::mma_commit(&ctl->bar);
  }
  if (!tc::mbar_wait_bounded(&ctl->bar, 1, kWaitLimit)) ctl->bad = 1;
  tc::fence_after_sync();
  // W^T rows (lane = key channel) and U^T rows (lane = value column), CW tokens a warp
  {
    uint32_t w0[16], u0[16];
    tc::tmem_ld16(tmem + la + 64 + CW * ch, w0);
    tc::tmem_ld16(tmem + la + 128 + CW * ch, u0);
    tc::tmem_wait_ld();
    float w[CW];
#pragma unroll
    for (int e = 0; e < CW; ++e) w[e] = tf32_nearest(__uint_as_float(w0[e]));
    float* wt = ws.WT + (unit * D + row) * C + CW * ch;
#pragma unroll
    for (int e = 0; e < CW; e += 4) *reinterpret_cast<float4*>(wt + e) = make_float4(w[e], w[e + 1], w[e + 2], w[e + 3]);
#pragma unroll
    for (int e = 0; e < CW; ++e) {
      const int64_t o = (unit * C + CW * ch + e) * D + row;
      ws.W[o] = w[e];
      ws.U[o] = __uint_as_float(u0[e]);
    }
  }
  {                                             // A_qk^T and T^T through a transposing stage
    float* const stg_a = reinterpret_cast<float*>(data + OPS);
    float* const stg_t = stg_a + C * (C + 1);
    for (int idx = tid; idx < C * C; idx += NT) {
      const int j = idx / C, i = idx % C;
      stg_a[i * (C + 1) + j] = tf32_nearest(s_Aq[j * CP + i]);
      stg_t[i * (C + 1) + j] = tf32_nearest(s_T[j * CP + i]);
    }
    __syncthreads();
    for (int idx = tid; idx < C * C; idx += NT) {
      const int i = idx / C, j = idx % C;
      ws.AqkT[unit * C * C + idx] = stg_a[i * (C + 1) + j];
      ws.TT[unit * C * C + idx] = stg_t[i * (C + 1) + j];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (ctl->bad && tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

cudaError_t launch_bwd_local_tc(const Problem& P, const SimtWorkspace& ws, ChunkWindow win, int slots,
                                bool perch, cudaStream_t st) {
  using namespace blt;
  if (slots <= 0) return cudaSuccess;
  auto k = perch ? bwd_local_tc_kernel<true> : bwd_local_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM));
  if (e != cudaSuccess) return e;
  k<<<dim3(static_cast<unsigned>(slots), P.HV), NT, SMEM, st>>>(P, ws, win);
  return cudaGetLastError();
}

cudaError_t launch_bwd_vc_tc(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A, ChunkWindow win,
                             int slots, cudaStream_t st) {
  using namespace bvt;
  if (slots <= 0) return cudaSuccess;
  const uint64_t units = static_cast<uint64_t>(slots) * static_cast<uint64_t>(P.HV);
  alignas(64) CUtensorMap tdo, tdy, ts, tds, te;
  if (!encode_f32_token_blocks(&tdo, A.d_o, static_cast<uint64_t>(P.T), static_cast<uint64_t>(P.HV), D, C) ||
      !encode_f32_blocks(&tdy, ws.dY, units * C, D, D, C) || !encode_f32_blocks(&ts, ws.Sck, units * D, D, D, D) ||
      !encode_f32_blocks(&tds, ws.dSck, units * D, D, D, D) || !encode_f32_blocks(&te, ws.E, units * C, D, D, C))
    return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(bwd_vc_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM));
  if (e != cudaSuccess) return e;
  bwd_vc_tc_kernel<<<dim3(static_cast<unsigned>(slots), P.HV), NT, SMEM, st>>>(P, ws, A, tdo, tdy, ts, tds, te, win);
  return cudaGetLastError();
}

}  // namespace kda
