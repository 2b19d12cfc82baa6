// backward.cu -- the backward pass of the chunkwise prefill, on CUDA cores in fp32.
//
// The chunk form of the forward pass ("You Could Have Come Up With Kimi Delta Attention",
// sec. 6: per chunk, with the incoming state S (stored d_k x d_v), K~ = k^ exp(G),
// Q~ = q^ exp(G), K_end = k^ exp(G_last - G), gamma = exp(G_last),
// L_im = sum_c k^_ic k^_mc exp(G_ic - G_mc) (m < i), M_im = sum_c q^_ic k^_mc exp(G_ic - G_mc)
// (m <= i), T = (I + diag(beta) L)^-1)
//
//     Y = diag(beta) (V - K~ S),   E = T Y,   O = Q~ S + M E,   S' = diag(gamma) S + K_end^T E
//
// is differentiated by the chain rule, chunk by chunk.  With dE = M^T dO + K_end dS' and
// dY = T^T dE:
//
//     dS  = Q~^T dO + diag(gamma) dS' - W^T dE          (W = T diag(beta) K~)
//     dV  = diag(beta) dY
//     dA  = -dY E^T (strictly lower),  dL = diag(beta) dA,   dM = dO E^T (lower)
//     dQ~ = dO S^T,  dK~ = -diag(beta) dY S^T,  dK_end = E dS'^T,  dgamma = rowsum(dS' * S)
//     dbeta_i = dY_i . (V - K~ S)_i + sum_m dA_im L_im
//
// and the pairwise products L and M, the decayed rows and gamma pass their gradients on to
// q^, k^ and the cumulative log-decay G, whose reverse cumulative sum is the gradient of g.
// The state recursion is the transpose of the forward chain, so it runs as a reverse scan over
// each sequence's chunks; everything else is chunk-parallel:
//
//   local   the forward's chunk-local stage, also keeping T and K~
//   scan    per (sequence, value head, value tile): forward over the chunks to record each
//           chunk's incoming state and E, then backward carrying dS: dE, dY, dV, dS per chunk
//   vc      per (chunk, value head): the contractions over the value dimension
//           (dQ~, dK~, dK_end, dA, dM, dgamma, the first term of dbeta)
//   pair    per (chunk, key head), over the value heads of its group: the pairwise terms,
//           dG and its reverse cumulative sum, dbeta, then the L2 normalisation's backward
//           and the sum over the group (GQA) for dq and dk
//
// The additive write (KDA_FLAG_NO_DELTA) has no L and no K~ S term: T = I, W = 0, and their
// gradient terms vanish.  The pairwise decay is evaluated per pair and channel, as in the
// CUDA-core forward, so no factor overflows.
#include <algorithm>

#include "backward.cuh"
#include "tc_utils.cuh"

namespace kda {

// Slots of the bounded workspace: a window of chunk positions holds every sequence's next
// `wc` chunks, wc = max(1, kBwdWindowSlots / (num_seqs * HV)) (so max(kBwdWindowSlots,
// num_seqs * HV) (chunk, value head) slots).
constexpr int kBwdWindowSlots = 512;

static int bwd_window_chunks(const Problem& P) {
  const int64_t pairs = static_cast<int64_t>(P.num_seqs) * P.HV;
  return static_cast<int>(std::max<int64_t>(1, kBwdWindowSlots / std::max<int64_t>(1, pairs)));
}

static bool bwd_tc(const Problem& P, bool qbf16) { return P.D == 128 && P.chunk == 64 && qbf16; }

// tc: the tensor-core kernels run (d = 128, chunk 64, bf16 inputs): the local stage keeps the
// transposed copies they read instead of Q~, A_qk and T.  wc > 0: the bounded workspace, the
// per-chunk arrays for one window's slots plus the checkpoints and the carried gradient.
static size_t bwd_layout(const Problem& P, char* base, BwdWorkspace* ws, bool tc, int wc) {
  size_t off = 0;
  PlanView pv;
  off = plan_layout(P, base, off, &pv);
  const int mc = plan_max_chunks(P);
  const size_t slots = wc > 0 ? static_cast<size_t>(P.num_seqs) * wc : static_cast<size_t>(mc);
  const size_t units = slots * P.HV;
  const size_t C = P.chunk, D = P.D;
  auto take = [&](size_t floats) -> float* {
    float* p = base ? reinterpret_cast<float*>(base + off) : nullptr;
    off += (floats * 4 + 255) & ~size_t(255);
    return p;
  };
  BwdWorkspace w{};
  w.loc.plan = pv;
  w.loc.W = take(units * C * D);
  w.loc.U = take(units * C * D);
  w.loc.Kend = take(units * C * D);
  w.loc.gamma = take(units * D);
  w.loc.Kt = take(units * C * D);
  if (tc) {
    w.loc.KendT = take(units * D * C);
    w.loc.QtT = take(units * D * C);
    w.loc.WT = take(units * D * C);
    w.loc.AqkT = take(units * C * C);
    w.loc.TT = take(units * C * C);
    w.loc.local_fb = reinterpret_cast<int32_t*>(take(units));
  } else {
    w.loc.Qt = take(units * C * D);
    w.loc.Aqk = take(units * C * C);
    w.loc.T = take(units * C * C);
  }
  w.Sck = take(units * D * D);
  w.dSck = take(units * D * D);
  w.E = take(units * C * D);
  w.dY = take(units * C * D);
  w.dQt = take(units * C * D);
  w.dKt = take(units * C * D);
  w.dKe = take(units * C * D);
  w.dA = take(units * C * C);
  w.dM = take(units * C * C);
  w.dgam = take(units * D);
  w.dbr = take(units * C);
  if (tc) w.pair_fb = reinterpret_cast<int32_t*>(take(slots * P.HK));
  if (wc > 0) {
    // checkpoint entries: sequence b's windows 1 .. ceil(n_b / wc) - 1 at c0_b / wc + w - 1,
    // disjoint between sequences and below max_chunks / wc
    w.ckpt = take(static_cast<size_t>(std::max(1, mc / wc)) * P.HV * D * D);
    w.carry = take(static_cast<size_t>(P.num_seqs) * P.HV * D * D);
  }
  if (ws) *ws = w;
  return off;
}

static int bwd_wc(const Problem& P, bool qbf16, bool compact) {
  return compact && bwd_tc(P, qbf16) ? bwd_window_chunks(P) : 0;
}

size_t bwd_workspace_bytes(const Problem& P, bool qbf16, bool compact) {
  return bwd_layout(P, nullptr, nullptr, bwd_tc(P, qbf16), bwd_wc(P, qbf16, compact));
}

// ------------------------------------------------------------------------------- scan

// The outputs of an R x BV product spread over the 256 threads as row segments: thread t owns
// row t / TPR and the JT consecutive columns from (t % TPR) * JT, so it keeps JT independent
// accumulators and reads operand rows as 16-byte vectors where JT allows.
template <int R, int BV>
struct RowTile {
  static constexpr int JT = R * BV / 256;
  static constexpr int TPR = BV / JT;
  static_assert(JT >= 1 && BV % JT == 0 && TPR * R == 256, "R x BV must tile 256 threads");
};

// A C x D fp32 matrix of the workspace into a shared buffer with rows of DP floats, as
// 16-byte asynchronous copies (committed as one group by the caller).
template <int C, int D, int DP>
__device__ __forceinline__ void mat_async(float* dst, const float* src, int tid) {
  for (int u = tid; u < C * D / 4; u += 256) {
    const int i = u / (D / 4), p4 = 4 * (u % (D / 4));
    tc::cp_async16(tc::smem_u32(dst + i * DP + p4), src + i * D + p4, 16);
  }
}

// Two chunk matrices in shared memory at a time (W and K_end going forward; K_end, then Q~ and
// W going back), the next one copied in while the current products run, and A_qk / T read
// through the L1 cache: 109 KB per CTA, two CTAs per SM.
template <int D, int C, int BV>
struct BwdScanSmem {
  static constexpr int DP = D + 4;   // padded rows: threads on different rows hit different banks
  static constexpr size_t floats = D * BV + 2 * C * DP + 3 * C * BV + D + C;
  static constexpr size_t bytes = floats * sizeof(float);
};

template <int D, int C, int BV, bool SBF16>
__global__ void __launch_bounds__(256, 2) bwd_scan_kernel(Problem P, BwdWorkspace ws, BwdArgs A) {
  constexpr int NT = 256;
  constexpr int DP = BwdScanSmem<D, C, BV>::DP;
  using TC = RowTile<C, BV>;        // the C x BV products
  using TD = RowTile<D, BV>;        // the D x BV products
  extern __shared__ __align__(16) float smem[];
  float* s_S = smem;                // [D][BV] state (forward) / its gradient (backward)
  float* s_A = s_S + D * BV;        // [C][DP] W (forward) / Q~ (backward)
  float* s_B = s_A + C * DP;        // [C][DP] K_end, then W (backward)
  float* s_X = s_B + C * DP;        // [C][BV] U (forward) / dO (backward)
  float* s_E = s_X + C * BV;        // [C][BV]
  float* s_dE = s_E + C * BV;       // [C][BV]
  float* s_g = s_dE + C * BV;       // [D] gamma
  float* s_b = s_g + D;             // [C] beta

  if (ws.loc.plan.info[1] == 0) return;
  const int HV = P.HV;
  const SeqHeadTile cta = seq_head_tile(ws.loc.plan, HV, D / BV);
  const int b = cta.b, h = cta.h, v0 = cta.vt * BV;
  const int tid = threadIdx.x;
  const int ri = tid / TC::TPR, rj = (tid % TC::TPR) * TC::JT;   // row segment of a C x BV product
  const int dc = tid / TD::TPR, dj = (tid % TD::TPR) * TD::JT;   // row segment of a D x BV product
  const int64_t sbase = (static_cast<int64_t>(P.slot_idx[b]) * HV + h) * D * D;
  for (int idx = tid; idx < D * BV; idx += NT) {
    const int c = idx / BV, j = idx % BV;
    s_S[idx] = SBF16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(P.pool)[sbase + c * D + v0 + j])
                     : static_cast<const float*>(P.pool)[sbase + c * D + v0 + j];
  }
  const int first = ws.loc.plan.seq_chunk0[b], last = ws.loc.plan.seq_chunk0[b + 1];
  auto cunit = [&](int cidx) { return static_cast<int64_t>(cidx) * HV + h; };
  // forward: record each chunk's incoming state and its corrected values E = U - W S
  if (first < last) {
    mat_async<C, D, DP>(s_A, ws.loc.W + cunit(first) * C * D, tid);
    mat_async<C, D, DP>(s_B, ws.loc.Kend + cunit(first) * C * D, tid);
    tc::cp_async_commit();
  }
  for (int cidx = first; cidx < last; ++cidx) {
    const int64_t unit = cunit(cidx);
    for (int idx = tid; idx < C * BV; idx += NT)
      s_X[idx] = ws.loc.U[unit * C * D + (idx / BV) * D + v0 + idx % BV];
    for (int c = tid; c < D; c += NT) s_g[c] = ws.loc.gamma[unit * D + c];
    for (int idx = tid; idx < D * BV; idx += NT)
      ws.Sck[unit * D * D + (idx / BV) * D + v0 + idx % BV] = s_S[idx];
    tc::cp_async_wait_all();
    __syncthreads();
    {
      float acc[TC::JT] = {};
      const float* w = s_A + ri * DP;
#pragma unroll 4
      for (int c = 0; c < D; ++c) {
        float x[TC::JT];
        ld_row(x, s_S + c * BV + rj);
        const float wc = w[c];
#pragma unroll
        for (int e = 0; e < TC::JT; ++e) acc[e] += wc * x[e];
      }
      float u[TC::JT];
      ld_row(u, s_X + ri * BV + rj);
#pragma unroll
      for (int e = 0; e < TC::JT; ++e) acc[e] = u[e] - acc[e];
      st_row(s_E + ri * BV + rj, acc);
      st_row(ws.E + unit * C * D + ri * D + v0 + rj, acc);
    }
    __syncthreads();
    if (cidx + 1 < last) {                      // W of the next chunk while the state updates
      mat_async<C, D, DP>(s_A, ws.loc.W + cunit(cidx + 1) * C * D, tid);
      tc::cp_async_commit();
    }
    {
      float acc[TD::JT];
      ld_row(acc, s_S + dc * BV + dj);
      const float gm = s_g[dc];
#pragma unroll
      for (int e = 0; e < TD::JT; ++e) acc[e] *= gm;
#pragma unroll 4
      for (int i = 0; i < C; ++i) {
        float x[TD::JT];
        ld_row(x, s_E + i * BV + dj);
        const float k = s_B[i * DP + dc];
#pragma unroll
        for (int e = 0; e < TD::JT; ++e) acc[e] += k * x[e];
      }
      st_row(s_S + dc * BV + dj, acc);
    }
    __syncthreads();
    if (cidx + 1 < last) {
      mat_async<C, D, DP>(s_B, ws.loc.Kend + cunit(cidx + 1) * C * D, tid);
      tc::cp_async_commit();
    }
  }
  // backward: dS starts as the gradient w.r.t. the final state
  for (int idx = tid; idx < D * BV; idx += NT)
    s_S[idx] = A.d_state ? A.d_state[sbase + (idx / BV) * D + v0 + idx % BV] : 0.f;
  if (first < last) {
    mat_async<C, D, DP>(s_B, ws.loc.Kend + cunit(last - 1) * C * D, tid);
    mat_async<C, D, DP>(s_A, ws.loc.Qt + cunit(last - 1) * C * D, tid);
    tc::cp_async_commit();
  }
  for (int cidx = last - 1; cidx >= first; --cidx) {
    const ChunkInfo ci = ws.loc.plan.chunks[cidx];
    const int64_t unit = cunit(cidx);
    const float* gM = ws.loc.Aqk + unit * C * C;
    const float* gT = ws.loc.T + unit * C * C;
    for (int idx = tid; idx < C * BV; idx += NT) {
      const int i = idx / BV, j = idx % BV;
      s_X[idx] = i < ci.n ? A.d_o[((ci.t0 + i) * HV + h) * D + v0 + j] : 0.f;
    }
    for (int c = tid; c < D; c += NT) s_g[c] = ws.loc.gamma[unit * D + c];
    for (int i = tid; i < C; i += NT) s_b[i] = i < ci.n ? P.beta[(ci.t0 + i) * HV + h] : 0.f;
    for (int idx = tid; idx < D * BV; idx += NT)
      ws.dSck[unit * D * D + (idx / BV) * D + v0 + idx % BV] = s_S[idx];
    tc::cp_async_wait_all();
    __syncthreads();
    {                                           // dE = A_qk^T dO + K_end dS'
      float acc[TC::JT] = {};
      for (int m = ri; m < C; ++m) {
        float x[TC::JT];
        ld_row(x, s_X + m * BV + rj);
        const float mm = __ldg(gM + m * C + ri);
#pragma unroll
        for (int e = 0; e < TC::JT; ++e) acc[e] += mm * x[e];
      }
      const float* k = s_B + ri * DP;
#pragma unroll 4
      for (int c = 0; c < D; ++c) {
        float x[TC::JT];
        ld_row(x, s_S + c * BV + rj);
        const float kc = k[c];
#pragma unroll
        for (int e = 0; e < TC::JT; ++e) acc[e] += kc * x[e];
      }
      st_row(s_dE + ri * BV + rj, acc);
    }
    __syncthreads();
    mat_async<C, D, DP>(s_B, ws.loc.W + unit * C * D, tid);   // K_end is done with
    tc::cp_async_commit();
    {                                           // dY = T^T dE, dV = diag(beta) dY
      float acc[TC::JT] = {};
      if (ri < ci.n) {
        for (int m = ri; m < C; ++m) {
          float x[TC::JT];
          ld_row(x, s_dE + m * BV + rj);
          const float t = __ldg(gT + m * C + ri);
#pragma unroll
          for (int e = 0; e < TC::JT; ++e) acc[e] += t * x[e];
        }
      }
      st_row(ws.dY + unit * C * D + ri * D + v0 + rj, acc);
      if (ri < ci.n) {
        const float bi = s_b[ri];
#pragma unroll
        for (int e = 0; e < TC::JT; ++e) acc[e] *= bi;
        st_row(A.dv + ((ci.t0 + ri) * HV + h) * D + v0 + rj, acc);
      }
    }
    // dS = diag(gamma) dS' + Q~^T dO - W^T dE: the Q~ part while W arrives
    float acc[TD::JT];
    ld_row(acc, s_S + dc * BV + dj);
    {
      const float gm = s_g[dc];
#pragma unroll
      for (int e = 0; e < TD::JT; ++e) acc[e] *= gm;
#pragma unroll 4
      for (int i = 0; i < C; ++i) {
        float x[TD::JT];
        ld_row(x, s_X + i * BV + dj);
        const float q = s_A[i * DP + dc];
#pragma unroll
        for (int e = 0; e < TD::JT; ++e) acc[e] += q * x[e];
      }
    }
    tc::cp_async_wait_all();
    __syncthreads();                            // W is in; Q~ is no longer read
    if (cidx - 1 >= first) {
      mat_async<C, D, DP>(s_A, ws.loc.Qt + cunit(cidx - 1) * C * D, tid);
      tc::cp_async_commit();
    }
#pragma unroll 4
    for (int i = 0; i < C; ++i) {
      float y[TD::JT];
      ld_row(y, s_dE + i * BV + dj);
      const float w = s_B[i * DP + dc];
#pragma unroll
      for (int e = 0; e < TD::JT; ++e) acc[e] -= w * y[e];
    }
    st_row(s_S + dc * BV + dj, acc);
    __syncthreads();                            // W is no longer read
    if (cidx - 1 >= first) {
      mat_async<C, D, DP>(s_B, ws.loc.Kend + cunit(cidx - 1) * C * D, tid);
      tc::cp_async_commit();
    }
  }
  tc::cp_async_wait_all();
  __syncthreads();
  if (A.d_state0)
    for (int idx = tid; idx < D * BV; idx += NT)
      A.d_state0[sbase + (idx / BV) * D + v0 + idx % BV] = s_S[idx];
}

// ------------------------------------------------------------------------------- vc

// Accumulators over the value dimension: thread t owns rows (t / 16) * C/16 + a (a < C/16)
// and, of a C x D product, columns (t % 16) * D/16 + b (b < D/16), of a C x C product
// columns (t % 16) * C/16 + b.
template <int D, int C, int BV>
struct BwdVcSmem {
  static constexpr int DP = D + 4, CP = C + 4;
  static constexpr size_t floats = C * DP + C + D * BV + 2 * BV * DP + 5 * C * BV + BV * CP;
  static constexpr size_t bytes = floats * sizeof(float);
};

template <int D, int C, int BV, bool QBF16>
__global__ void __launch_bounds__(256) bwd_vc_kernel(Problem P, BwdWorkspace ws, BwdArgs A, ChunkWindow win) {
  constexpr int NT = 256;
  constexpr int DP = BwdVcSmem<D, C, BV>::DP, CP = BwdVcSmem<D, C, BV>::CP;
  constexpr int IR = C / 16, JC = D / 16, JM = C / 16;
  using TC = RowTile<C, BV>;
  extern __shared__ __align__(16) float smem[];
  float* s_Kt = smem;               // [C][DP] K~
  float* s_b = s_Kt + C * DP;       // [C]
  float* s_S = s_b + C;             // [D][BV] S tile
  float* s_St = s_S + D * BV;       // [BV][DP] S tile, transposed
  float* s_dSt = s_St + BV * DP;    // [BV][DP] dS' tile, transposed
  float* s_V = s_dSt + BV * DP;     // [C][BV]
  float* s_E = s_V + C * BV;        // [C][BV]
  float* s_dO = s_E + C * BV;       // [C][BV]
  float* s_dY = s_dO + C * BV;      // [C][BV]
  float* s_R = s_dY + C * BV;       // [C][BV] V - K~ S
  float* s_Et = s_R + C * BV;       // [BV][CP]

  int gc;
  if (ws.loc.plan.info[1] == 0 || !window_chunk(ws.loc.plan, P.num_seqs, win, blockIdx.x, &gc)) return;
  const ChunkInfo ci = ws.loc.plan.chunks[gc];
  const int h = blockIdx.y, HV = P.HV, tid = threadIdx.x;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * HV + h;
  const bool delta = !(P.flags & KDA_FLAG_NO_DELTA);
  const int ri = tid / TC::TPR, rj = (tid % TC::TPR) * TC::JT;
  const int r0 = (tid / 16) * IR, c0 = (tid % 16) * JC, m0 = (tid % 16) * JM;
  for (int idx = tid; idx < C * D; idx += NT) s_Kt[(idx / D) * DP + idx % D] = ws.loc.Kt[unit * C * D + idx];
  for (int i = tid; i < C; i += NT) s_b[i] = i < ci.n ? P.beta[(ci.t0 + i) * HV + h] : 0.f;

  float aQ[IR][JC], aK[IR][JC], aE[IR][JC], aA[IR][JM], aM[IR][JM];
#pragma unroll
  for (int a = 0; a < IR; ++a) {
#pragma unroll
    for (int b = 0; b < JC; ++b) aQ[a][b] = aK[a][b] = aE[a][b] = 0.f;
#pragma unroll
    for (int b = 0; b < JM; ++b) aA[a][b] = aM[a][b] = 0.f;
  }
  float gam_acc = 0.f, br_acc = 0.f;

  for (int v0 = 0; v0 < D; v0 += BV) {
    __syncthreads();
    for (int idx = tid; idx < D * BV; idx += NT) {
      const int c = idx / BV, j = idx % BV;
      const float sv = ws.Sck[unit * D * D + c * D + v0 + j];
      s_S[idx] = sv;
      s_St[j * DP + c] = sv;
      s_dSt[j * DP + c] = ws.dSck[unit * D * D + c * D + v0 + j];
    }
    for (int idx = tid; idx < C * BV; idx += NT) {
      const int i = idx / BV, j = idx % BV;
      const bool live = i < ci.n;
      s_V[idx] = live ? load_elem<QBF16>(P.v, (ci.t0 + i) * P.v_stride + static_cast<int64_t>(h) * D + v0 + j) : 0.f;
      const float e = ws.E[unit * C * D + i * D + v0 + j];
      s_E[idx] = e;
      s_Et[j * CP + i] = e;
      s_dY[idx] = ws.dY[unit * C * D + i * D + v0 + j];
      s_dO[idx] = live ? A.d_o[((ci.t0 + i) * HV + h) * D + v0 + j] : 0.f;
    }
    __syncthreads();
    {                                           // R = V - K~ S
      float ks[TC::JT] = {};
      if (delta) {
        const float* kt = s_Kt + ri * DP;
#pragma unroll 4
        for (int c = 0; c < D; ++c) {
          float x[TC::JT];
          ld_row(x, s_S + c * BV + rj);
          const float kc = kt[c];
#pragma unroll
          for (int e = 0; e < TC::JT; ++e) ks[e] += kc * x[e];
        }
      }
      float v[TC::JT];
      ld_row(v, s_V + ri * BV + rj);
#pragma unroll
      for (int e = 0; e < TC::JT; ++e) v[e] -= ks[e];
      st_row(s_R + ri * BV + rj, v);
    }
    __syncthreads();
#pragma unroll 2
    for (int j = 0; j < BV; ++j) {
      float xo[IR], xy[IR], xe[IR], st[JC], dst[JC], et[JM];
#pragma unroll
      for (int a = 0; a < IR; ++a) {
        xo[a] = s_dO[(r0 + a) * BV + j];
        xy[a] = s_dY[(r0 + a) * BV + j];
        xe[a] = s_E[(r0 + a) * BV + j];
      }
      ld_row(st, s_St + j * DP + c0);
      ld_row(dst, s_dSt + j * DP + c0);
      ld_row(et, s_Et + j * CP + m0);
#pragma unroll
      for (int a = 0; a < IR; ++a) {
#pragma unroll
        for (int b = 0; b < JC; ++b) {
          aQ[a][b] += xo[a] * st[b];
          aK[a][b] += xy[a] * st[b];
          aE[a][b] += xe[a] * dst[b];
        }
#pragma unroll
        for (int b = 0; b < JM; ++b) {
          aA[a][b] += xy[a] * et[b];
          aM[a][b] += xo[a] * et[b];
        }
      }
    }
    if (tid < D)
      for (int j = 0; j < BV; ++j) gam_acc += s_dSt[j * DP + tid] * s_St[j * DP + tid];
    if (tid < C)
      for (int j = 0; j < BV; ++j) {
        const int jj = (j + tid) % BV;          // rotated start: rows of one warp hit different banks
        br_acc += s_dY[tid * BV + jj] * s_R[tid * BV + jj];
      }
  }
#pragma unroll
  for (int a = 0; a < IR; ++a) {
    const int i = r0 + a;
    const float nb = delta ? -s_b[i] : 0.f;
    float k[JC];
#pragma unroll
    for (int b = 0; b < JC; ++b) k[b] = nb * aK[a][b];
    st_row(ws.dQt + unit * C * D + i * D + c0, aQ[a]);
    st_row(ws.dKt + unit * C * D + i * D + c0, k);
    st_row(ws.dKe + unit * C * D + i * D + c0, aE[a]);
    float da[JM], dm[JM];
#pragma unroll
    for (int b = 0; b < JM; ++b) {
      const int m = m0 + b;
      da[b] = (delta && m < i) ? -aA[a][b] : 0.f;
      dm[b] = m <= i ? aM[a][b] : 0.f;
    }
    st_row(ws.dA + unit * C * C + i * C + m0, da);
    st_row(ws.dM + unit * C * C + i * C + m0, dm);
  }
  if (tid < D) ws.dgam[unit * D + tid] = gam_acc;
  if (tid < C) ws.dbr[unit * C + tid] = br_acc;
}

// ------------------------------------------------------------------------------- pair

// Thread t owns the entries (r0 + a, c0 + b) of every C x D quantity, r0 = (t / 16) * C/16,
// c0 = (t % 16) * D/16 (a < C/16, b < D/16): a row group is one half-warp.  The pairwise
// products are then small matrix products, P1 = (dM o X) k^, P2 = (dA o X) k^,
// P3 = (dM o X)^T q^ + (diag(beta) dA o X)^T k^ with X the pairwise decay, which for scalar
// decay is folded into dM and dA once per chunk.
template <int D, int C, bool PERCH>
struct BwdPairSmem {
  static constexpr int GW = PERCH ? D : 1;
  static constexpr int DP = D + 4, CP = C + 4;
  static constexpr size_t floats =
      3 * C * DP + C * GW + 2 * C * CP + 6 * C + 3 * D + (PERCH ? C * DP : 0);
  static constexpr size_t bytes = floats * sizeof(float);
};


template <int D, int C, bool QBF16, bool PERCH>
__global__ void __launch_bounds__(256) bwd_pair_kernel(Problem P, BwdWorkspace ws, BwdArgs A, ChunkWindow win,
                                                        int fb_only) {
  constexpr int NT = 256;
  constexpr int IR = C / 16, JC = D / 16;
  constexpr int GW = BwdPairSmem<D, C, PERCH>::GW;
  constexpr int DP = BwdPairSmem<D, C, PERCH>::DP, CP = BwdPairSmem<D, C, PERCH>::CP;
  extern __shared__ __align__(16) float smem[];
  float* s_q = smem;               // [C][DP] q^ = s q / |q| (scaled)
  float* s_k = s_q + C * DP;       // [C][DP] k^ = k / |k|
  float* s_dG = s_k + C * DP;      // [C][DP] gradient w.r.t. G, one value head at a time
  float* s_G = s_dG + C * DP;      // [C][GW] cumulative log-decay
  float* s_dA = s_G + C * GW;      // [C][CP] dA (times the pairwise decay for scalar decay)
  float* s_dM = s_dA + C * CP;     // [C][CP] dM (likewise)
  float* s_b = s_dM + C * CP;      // [C] beta
  float* s_rq = s_b + C;           // [C] 1/|q| (1 without the norm)
  float* s_rk = s_rq + C;          // [C]
  float* s_db = s_rk + C;          // [C] pairwise part of dbeta
  float* s_dotq = s_db + C;        // [C]
  float* s_dotk = s_dotq + C;      // [C]
  float* s_dGl = s_dotk + C;       // [D] gradient w.r.t. G_last
  float* s_gam = s_dGl + D;        // [D]
  float* s_ga = s_gam + D;         // [D] G at the chunk's middle token (per-channel decay)
  float* s_E = s_ga + D;           // [C][DP] exp(G - G_a) (per-channel decay, anchored)

  int gc;
  if (ws.loc.plan.info[1] == 0 || !window_chunk(ws.loc.plan, P.num_seqs, win, blockIdx.x, &gc)) return;
  // after the tensor-core kernel: only the (chunk, key head) pairs it left here
  if (fb_only && ws.pair_fb[static_cast<int64_t>(blockIdx.x) * P.HK + blockIdx.y] == 0) return;
  const ChunkInfo ci = ws.loc.plan.chunks[gc];
  const int kh = blockIdx.y, HV = P.HV, ratio = HV / P.HK, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool delta = !(P.flags & KDA_FLAG_NO_DELTA);
  const int n = ci.n;
  const int r0 = (tid / 16) * IR, c0 = (tid % 16) * JC;
  const bool lead = (tid % 16) == 0;         // writes its half-warp's row sums

  for (int idx = tid; idx < C * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    const bool live = i < n;
    s_q[i * DP + c] = live ? load_elem<QBF16>(P.q, (ci.t0 + i) * P.q_stride + static_cast<int64_t>(kh) * D + c) : 0.f;
    s_k[i * DP + c] = live ? load_elem<QBF16>(P.k, (ci.t0 + i) * P.k_stride + static_cast<int64_t>(kh) * D + c) : 0.f;
  }
  __syncthreads();
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

  for (int h = kh * ratio; h < (kh + 1) * ratio; ++h) {
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * HV + h;
    __syncthreads();
    // cumulative log-decay (padded rows add nothing), beta, dA, dM: the log-decay rows are
    // loaded by all threads at once, then summed down the rows in shared memory
    for (int idx = tid; idx < C * GW; idx += NT) {
      const int i = idx / GW, c = idx % GW;
      s_G[idx] = i < n ? (PERCH ? P.g[((ci.t0 + i) * HV + h) * D + c] : P.g[(ci.t0 + i) * HV + h]) : 0.f;
    }
    __syncthreads();
    for (int c = tid; c < GW; c += NT) {
      float acc = 0.f;
      for (int i = 0; i < C; ++i) {
        acc += s_G[i * GW + c];
        s_G[i * GW + c] = acc;
      }
    }
    for (int i = tid; i < C; i += NT) s_b[i] = i < n ? P.beta[(ci.t0 + i) * HV + h] : 0.f;
    for (int idx = tid; idx < C * C; idx += NT) {
      s_dA[(idx / C) * CP + idx % C] = ws.dA[unit * C * C + idx];
      s_dM[(idx / C) * CP + idx % C] = ws.dM[unit * C * C + idx];
    }
    for (int c = tid; c < D; c += NT) s_dGl[c] = 0.f;
    __syncthreads();
    for (int c = tid; c < D; c += NT) s_gam[c] = expf(s_G[(C - 1) * GW + (PERCH ? c : 0)]);
    if constexpr (!PERCH) {                     // fold exp(G_i - G_m) into the lower triangles
      for (int idx = tid; idx < C * C; idx += NT) {
        const int i = idx / C, m = idx % C;
        const float x = m <= i ? expf(s_G[i] - s_G[m]) : 0.f;
        s_dA[i * CP + m] *= x;
        s_dM[i * CP + m] *= x;
      }
      __syncthreads();
    }
    // per-channel decay: the pairwise factor exp(G_ic - G_mc) = E+_ic / E+_mc with
    // E+ = exp(G - G_a) (anchor at the middle token) while the decay stays in range; then
    // P1, P2 = E+ (dM, dA) K- with K- = k^ / E+ and P3 = (dM^T (q^ E+) + ...)/E+, no exp per pair
    bool anch = false;
    if constexpr (PERCH) {
      const int am = (n - 1) / 2;
      for (int c = tid; c < D; c += NT) s_ga[c] = s_G[am * GW + c];
      __syncthreads();
      bool wide = false;
      for (int idx = tid; idx < C * D; idx += NT) {
        const int i = idx / D, c = idx % D;
        wide |= fabsf(s_G[i * GW + c] - s_ga[c]) > kSimtAnchorRange;
      }
      anch = !__syncthreads_or(wide);
      if (anch) {
        for (int idx = tid; idx < C * D; idx += NT) {
          const int i = idx / D, c = idx % D;
          const float d = s_G[i * GW + c] - s_ga[c];
          s_E[i * DP + c] = expf(d);
          s_dG[i * DP + c] = s_k[i * DP + c] * expf(-d);     // K-, until dG is formed
        }
        __syncthreads();
      }
    }
    float p1[IR][JC], p2[IR][JC], p3[IR][JC];
#pragma unroll
    for (int a = 0; a < IR; ++a)
#pragma unroll
      for (int b = 0; b < JC; ++b) p1[a][b] = p2[a][b] = p3[a][b] = 0.f;
    if (PERCH && anch) {
      for (int m = 0; m < r0 + IR; ++m) {
        float km[JC];
        ld_row(km, s_dG + m * DP + c0);
#pragma unroll
        for (int a = 0; a < IR; ++a) {
          const int i = r0 + a;
          if (m > i) continue;
          const float fm = s_dM[i * CP + m], fa = s_dA[i * CP + m];
#pragma unroll
          for (int b = 0; b < JC; ++b) {
            p1[a][b] += fm * km[b];
            p2[a][b] += fa * km[b];
          }
        }
      }
      for (int m = r0; m < C; ++m) {
        float qm[JC], km[JC], em[JC];
        ld_row(qm, s_q + m * DP + c0);
        ld_row(km, s_k + m * DP + c0);
        ld_row(em, s_E + m * DP + c0);
        const float bm = delta ? s_b[m] : 0.f;
#pragma unroll
        for (int a = 0; a < IR; ++a) {
          const int i = r0 + a;
          if (m < i) continue;
          const float fm = s_dM[m * CP + i], fa = bm * s_dA[m * CP + i];
#pragma unroll
          for (int b = 0; b < JC; ++b) p3[a][b] += (fm * qm[b] + fa * km[b]) * em[b];
        }
      }
#pragma unroll
      for (int a = 0; a < IR; ++a)
#pragma unroll
        for (int b = 0; b < JC; ++b) {
          const int i = r0 + a, c = c0 + b;
          const float d = s_G[i * GW + c] - s_ga[c];
          const float ep = s_E[i * DP + c];
          p1[a][b] *= ep;
          p2[a][b] *= ep;
          p3[a][b] *= expf(-d);
        }
    } else {
      // the entry as the row: P1 = sum_{m<=i} dM_im x_imc k^_mc, P2 = sum_{m<i} dA_im x_imc k^_mc
      for (int m = 0; m < r0 + IR; ++m) {
        float km[JC];
        ld_row(km, s_k + m * DP + c0);
#pragma unroll
        for (int a = 0; a < IR; ++a) {
          const int i = r0 + a;
          if (m > i) continue;
          const float fm = s_dM[i * CP + m], fa = s_dA[i * CP + m];
#pragma unroll
          for (int b = 0; b < JC; ++b) {
            const float kd = PERCH ? km[b] * expf(s_G[i * GW + c0 + b] - s_G[m * GW + c0 + b]) : km[b];
            p1[a][b] += fm * kd;
            p2[a][b] += fa * kd;
          }
        }
      }
      // the entry as the column: P3 = sum_{m>=i} dM_mi x_mic q^_mc + sum_{m>i} beta_m dA_mi x_mic k^_mc
      for (int m = r0; m < C; ++m) {
        float qm[JC], km[JC];
        ld_row(qm, s_q + m * DP + c0);
        ld_row(km, s_k + m * DP + c0);
        const float bm = delta ? s_b[m] : 0.f;
#pragma unroll
        for (int a = 0; a < IR; ++a) {
          const int i = r0 + a;
          if (m < i) continue;
          const float fm = s_dM[m * CP + i], fa = bm * s_dA[m * CP + i];
#pragma unroll
          for (int b = 0; b < JC; ++b) {
            const float x = fm * qm[b] + fa * km[b];
            p3[a][b] += PERCH ? x * expf(s_G[m * GW + c0 + b] - s_G[i * GW + c0 + b]) : x;
          }
        }
      }
    }
    __syncthreads();                            // K- (in s_dG) is read no more
    float gl[JC];
#pragma unroll
    for (int b = 0; b < JC; ++b) gl[b] = 0.f;
#pragma unroll
    for (int a = 0; a < IR; ++a) {
      const int i = r0 + a;
      float dqt[JC], dkt[JC], dke[JC];
      ld_row(dqt, ws.dQt + unit * C * D + i * D + c0);
      ld_row(dkt, ws.dKt + unit * C * D + i * D + c0);
      ld_row(dke, ws.dKe + unit * C * D + i * D + c0);
      const float bi = s_b[i];
      float bl = 0.f;
#pragma unroll
      for (int b = 0; b < JC; ++b) {
        const int gc = PERCH ? c0 + b : 0;
        const float Gi = s_G[i * GW + gc], Gl = s_G[(C - 1) * GW + gc];
        const float eG = expf(Gi), eL = expf(Gl - Gi);
        const float qv = s_q[i * DP + c0 + b], kv = s_k[i * DP + c0 + b];
        adq[a][b] += p1[a][b] + dqt[b] * eG;
        adk[a][b] += bi * p2[a][b] + p3[a][b] + dkt[b] * eG + dke[b] * eL;
        s_dG[i * DP + c0 + b] = qv * p1[a][b] + kv * bi * p2[a][b] - kv * p3[a][b] +
                                dqt[b] * qv * eG + dkt[b] * kv * eG - dke[b] * kv * eL;
        bl += kv * p2[a][b];                    // dbeta's pairwise part: sum_c k^_ic P2_ic
        gl[b] += dke[b] * kv * eL;              // K_end's path into G_last
      }
      bl = halfwarp_sum(bl);
      if (lead) s_db[i] = bl;
    }
#pragma unroll
    for (int b = 0; b < JC; ++b) atomicAdd(&s_dGl[c0 + b], gl[b]);
    __syncthreads();
    for (int c = tid; c < D; c += NT)
      s_dG[(C - 1) * DP + c] += s_dGl[c] + ws.dgam[unit * D + c] * s_gam[c];
    __syncthreads();
    // dg = reverse cumulative sum of dG over the chunk's rows
    if (PERCH) {
      for (int c = tid; c < D; c += NT) {
        float acc = 0.f;
        for (int i = C - 1; i >= 0; --i) {
          acc += s_dG[i * DP + c];
          if (i < n) A.dg[((ci.t0 + i) * HV + h) * D + c] = acc;
        }
      }
    } else {
      for (int i = warp; i < C; i += NT / 32) {
        float sm = 0.f;
        for (int c = lane; c < D; c += 32) sm += s_dG[i * DP + c];
        sm = warp_sum(sm);
        if (lane == 0) s_dotq[i] = sm;
      }
      __syncthreads();
      if (tid == 0) {
        float acc = 0.f;
        for (int i = C - 1; i >= 0; --i) {
          acc += s_dotq[i];
          if (i < n) A.dg[(ci.t0 + i) * HV + h] = acc;
        }
      }
    }
    for (int i = tid; i < n; i += NT)
      A.dbeta[(ci.t0 + i) * HV + h] = ws.dbr[unit * C + i] + (delta ? s_db[i] : 0.f);
  }
  // the L2 normalisation's backward: with u = x / |x|, dx = (du - u (u . du)) / |x|
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
    const float inv_s = 1.f / P.scale;
    if (i >= n) continue;
    float oq[JC], ok[JC];
#pragma unroll
    for (int b = 0; b < JC; ++b) {
      if (P.l2norm) {
        // q^ = s u_q with u_q = q / |q|: dq = s (dq^ - u_q (u_q . dq^)) / |q|
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

// ------------------------------------------------------------------------------- launch

template <typename K>
static cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <int D, int C, bool QBF16, bool PERCH, bool SBF16>
static cudaError_t launch_bwd_t(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A, int wc,
                                cudaStream_t st) {
  constexpr int BV = D >= 32 ? 32 : D;
  // bf16 inputs at d = 128, chunk 64: the scans and the value-dimension contractions on tensor
  // cores (tf32 operands; the fp32 inputs' tighter bound keeps them on CUDA cores)
  constexpr bool kTc = D == 128 && C == 64 && QBF16;
  cudaError_t e;
  auto lk = simt_local_kernel<D, C, QBF16, PERCH>;
  if ((e = set_smem(lk, SimtLocalSmem<D, C>::bytes)) != cudaSuccess) return e;
  auto sk = bwd_scan_kernel<D, C, BV, SBF16>;
  if ((e = set_smem(sk, BwdScanSmem<D, C, BV>::bytes)) != cudaSuccess) return e;
  auto vk = bwd_vc_kernel<D, C, BV, QBF16>;
  if ((e = set_smem(vk, BwdVcSmem<D, C, BV>::bytes)) != cudaSuccess) return e;
  auto pk = bwd_pair_kernel<D, C, QBF16, PERCH>;
  if ((e = set_smem(pk, BwdPairSmem<D, C, PERCH>::bytes)) != cudaSuccess) return e;
  // the chunk-parallel kernels of one window (or of every chunk: wc == 0)
  auto local = [&](ChunkWindow win, int slots) -> cudaError_t {
    if (slots <= 0) return cudaSuccess;
    if (kTc) {
      cudaError_t r = launch_bwd_local_tc(P, ws.loc, win, slots, PERCH, st);
      if (r != cudaSuccess || !PERCH) return r;
      // per-channel decay: the chunks outside the anchored factors' range, exactly
      lk<<<dim3(slots, P.HV), 256, SimtLocalSmem<D, C>::bytes, st>>>(P, ws.loc, win, 1);
      return cudaGetLastError();
    }
    lk<<<dim3(slots, P.HV), 256, SimtLocalSmem<D, C>::bytes, st>>>(P, ws.loc, win, 0);
    return cudaGetLastError();
  };
  auto contractions = [&](ChunkWindow win, int slots) -> cudaError_t {
    if (slots <= 0) return cudaSuccess;
    cudaError_t r = kTc ? launch_bwd_vc_tc(P, ws, A, win, slots, st) : cudaErrorNotSupported;
    if (r == cudaErrorNotSupported) {
      vk<<<dim3(slots, P.HV), 256, BwdVcSmem<D, C, BV>::bytes, st>>>(P, ws, A, win);
      r = cudaGetLastError();
    }
    if (r != cudaSuccess) return r;
    if (kTc) {
      r = launch_bwd_pair_tc(P, ws, A, win, slots, PERCH, st);
      if (r != cudaSuccess || !PERCH) return r;
      // per-channel decay: the chunks outside the anchored factors' range, exactly
      pk<<<dim3(slots, P.HK), 256, BwdPairSmem<D, C, PERCH>::bytes, st>>>(P, ws, A, win, 1);
      return cudaGetLastError();
    }
    pk<<<dim3(slots, P.HK), 256, BwdPairSmem<D, C, PERCH>::bytes, st>>>(P, ws, A, win, 0);
    return cudaGetLastError();
  };
  if (wc == 0) {
    const int mc = plan_max_chunks(P);
    const ChunkWindow all{0, 0};
    if ((e = local(all, mc)) != cudaSuccess) return e;
    if (kTc) {
      e = launch_bwd_scans_tc(P, ws, A, SBF16, all, mc, true, st);
    } else {
      sk<<<seq_head_tile_ctas(P, D / BV), 256, BwdScanSmem<D, C, BV>::bytes, st>>>(P, ws, A);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    return contractions(all, mc);
  }
  if (!kTc) return cudaErrorNotSupported;
  // bounded workspace: the longest sequence sets the number of windows (one read of the
  // chunk table's summary), a forward sweep stores each window's entering state, and the
  // backward sweep reruns each window from its checkpoint, latest window first
  int32_t longest = 0;
  if ((e = cudaMemcpyAsync(&longest, ws.loc.plan.info + 2, sizeof(int32_t), cudaMemcpyDeviceToHost, st)) !=
          cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return e;
  const int nw = std::max(1, (longest + wc - 1) / wc);
  const int slots = P.num_seqs * wc;
  for (int w = 0; w + 1 < nw; ++w) {
    const ChunkWindow win{w, wc};
    if ((e = local(win, slots)) != cudaSuccess) return e;
    if ((e = launch_bwd_scans_tc(P, ws, A, SBF16, win, slots, false, st)) != cudaSuccess) return e;
  }
  for (int w = nw - 1; w >= 0; --w) {
    const ChunkWindow win{w, wc};
    if ((e = local(win, slots)) != cudaSuccess) return e;
    if ((e = launch_bwd_scans_tc(P, ws, A, SBF16, win, slots, true, st)) != cudaSuccess) return e;
    if ((e = contractions(win, slots)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D, int C>
static cudaError_t launch_bwd_dc(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A,
                                 bool q, bool pc, bool sb, int wc, cudaStream_t st) {
  if (q) {
    if (pc) return sb ? launch_bwd_t<D, C, true, true, true>(P, ws, A, wc, st)
                      : launch_bwd_t<D, C, true, true, false>(P, ws, A, wc, st);
    return sb ? launch_bwd_t<D, C, true, false, true>(P, ws, A, wc, st)
              : launch_bwd_t<D, C, true, false, false>(P, ws, A, wc, st);
  }
  if (pc) return sb ? launch_bwd_t<D, C, false, true, true>(P, ws, A, wc, st)
                    : launch_bwd_t<D, C, false, true, false>(P, ws, A, wc, st);
  return sb ? launch_bwd_t<D, C, false, false, true>(P, ws, A, wc, st)
            : launch_bwd_t<D, C, false, false, false>(P, ws, A, wc, st);
}

template <int D>
static cudaError_t launch_bwd_d(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A,
                                bool q, bool pc, bool sb, int wc, cudaStream_t st) {
  switch (P.chunk) {
    case 16: return launch_bwd_dc<D, 16>(P, ws, A, q, pc, sb, wc, st);
    case 32: return launch_bwd_dc<D, 32>(P, ws, A, q, pc, sb, wc, st);
    default: return launch_bwd_dc<D, 64>(P, ws, A, q, pc, sb, wc, st);
  }
}

cudaError_t launch_prefill_bwd(const Problem& P, void* workspace, const float* d_o,
                               const float* d_state, float* dq, float* dk, float* dv,
                               float* dbeta, float* dg, float* d_state0, bool qbf16, bool perch,
                               bool sbf16, bool compact, cudaStream_t stream) {
  BwdWorkspace ws;
  const int wc = bwd_wc(P, qbf16, compact);
  bwd_layout(P, static_cast<char*>(workspace), &ws, bwd_tc(P, qbf16), wc);
  const BwdArgs A{d_o, d_state, dq, dk, dv, dbeta, dg, d_state0};
  cudaError_t e = launch_plan(P, ws.loc.plan, stream);
  if (e != cudaSuccess) return e;
  if (P.D == 128) return launch_bwd_d<128>(P, ws, A, qbf16, perch, sbf16, wc, stream);
  return launch_bwd_d<16>(P, ws, A, qbf16, perch, sbf16, wc, stream);
}

}  // namespace kda
