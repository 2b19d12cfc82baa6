// prefill_simt.cu -- chunkwise prefill on CUDA cores, fp32 throughout.
//
// This is the exact-arithmetic path: fp32 inputs (and any head size the
// library supports) run here, and it is the schedule the tensor-core path
// reproduces with lower-precision operands.  Stages, per the chunkwise
// derivation ("You Could Have Come Up With Kimi Delta Attention", sec. 6 and
// the pipeline of sec. 6.6; "From Attention to Learned Memory", sec. 4):
//
//   plan    ragged offsets -> chunk table (chunks restart at every sequence)
//   local   per (chunk, value head), all chunks in parallel:
//             L2 norm of q and k, query scale, in-chunk cumulative log-decay G;
//             A_kk[i][j] = beta_i sum_c k_i k_j exp(G_i - G_j)      (j < i)
//             A_qk[i][j] =        sum_c q_i k_j exp(G_i - G_j)      (j <= i)
//             T = (I + A_kk)^-1 by forward substitution on 16x16 diagonal
//               blocks, then merges T21 = -T22 A21 T11 up to the chunk;
//             W = T diag(beta) (k exp(G)),  U = T diag(beta) v,
//             Q~ = q exp(G),  K_end = k exp(G_last - G),  gamma = exp(G_last)
//   scan    per (sequence, value head, value tile), sequential over chunks:
//             E = U - W S,  O = Q~ S + A_qk E,  S = diag(gamma) S + K_end^T E
//           (S is the stored d_k x d_v state), then S goes back to its slot.
//
// The pairwise decay exp(G_i - G_j) is evaluated per pair and channel, so no
// factor can overflow whatever the decay.
#include "prefill_simt.cuh"

namespace kda {

static size_t simt_layout(const Problem& P, char* base, SimtWorkspace* ws) {
  size_t off = 0;
  PlanView pv;
  off = plan_layout(P, base, off, &pv);
  const size_t mc = static_cast<size_t>(plan_max_chunks(P));
  const size_t units = mc * P.HV;
  const size_t C = P.chunk, D = P.D;
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? base + off : nullptr;
    off += (bytes + 255) & ~size_t(255);
    return p;
  };
  float* W = reinterpret_cast<float*>(take(units * C * D * 4));
  float* U = reinterpret_cast<float*>(take(units * C * D * 4));
  float* Qt = reinterpret_cast<float*>(take(units * C * D * 4));
  float* Kend = reinterpret_cast<float*>(take(units * C * D * 4));
  float* Aqk = reinterpret_cast<float*>(take(units * C * C * 4));
  float* gamma = reinterpret_cast<float*>(take(units * D * 4));
  if (ws) *ws = SimtWorkspace{pv, W, U, Qt, Kend, Aqk, gamma, nullptr, nullptr};
  return off;
}

size_t simt_workspace_bytes(const Problem& P) { return simt_layout(P, nullptr, nullptr); }

template <int D, int C, int BV>
struct SimtScanSmem {
  static constexpr size_t floats = D * BV + 3 * C * D + 2 * C * BV + C * C + D;
  static constexpr size_t bytes = floats * sizeof(float);
};

template <int D, int C, int BV, bool SBF16>
__global__ void __launch_bounds__(256) simt_scan_kernel(Problem P, SimtWorkspace ws) {
  constexpr int NT = 256;
  extern __shared__ float smem[];
  float* s_S = smem;              // [D][BV] state tile (stored orientation)
  float* s_W = s_S + D * BV;      // [C][D]
  float* s_Q = s_W + C * D;       // [C][D]
  float* s_K = s_Q + C * D;       // [C][D]
  float* s_U = s_K + C * D;       // [C][BV]
  float* s_E = s_U + C * BV;      // [C][BV]
  float* s_A = s_E + C * BV;      // [C][C]
  float* s_g = s_A + C * C;       // [D]

  if (ws.plan.info[1] == 0) return;
  const int HV = P.HV;
  const SeqHeadTile cta = seq_head_tile(ws.plan, HV, D / BV);
  const int b = cta.b, h = cta.h, v0 = cta.vt * BV;
  const int tid = threadIdx.x;
  const uint32_t bos = P.offsets[b], eos = P.offsets[b + 1];
  if (eos <= bos) return;
  const int64_t sbase = (static_cast<int64_t>(P.slot_idx[b]) * HV + h) * D * D;
  for (int idx = tid; idx < D * BV; idx += NT) {
    const int c = idx / BV, j = idx % BV;
    s_S[idx] = SBF16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(P.pool)[sbase + c * D + v0 + j])
                     : static_cast<const float*>(P.pool)[sbase + c * D + v0 + j];
  }
  const int first = ws.plan.seq_chunk0[b], last = ws.plan.seq_chunk0[b + 1];
  for (int cidx = first; cidx < last; ++cidx) {
    const ChunkInfo ci = ws.plan.chunks[cidx];
    const int64_t unit = static_cast<int64_t>(cidx) * HV + h;
    for (int idx = tid; idx < C * D; idx += NT) {
      s_W[idx] = ws.W[unit * C * D + idx];
      s_Q[idx] = ws.Qt[unit * C * D + idx];
      s_K[idx] = ws.Kend[unit * C * D + idx];
    }
    for (int idx = tid; idx < C * BV; idx += NT)
      s_U[idx] = ws.U[unit * C * D + (idx / BV) * D + v0 + idx % BV];
    for (int idx = tid; idx < C * C; idx += NT) s_A[idx] = ws.Aqk[unit * C * C + idx];
    for (int c = tid; c < D; c += NT) s_g[c] = ws.gamma[unit * D + c];
    __syncthreads();
    // E = U - W S
    for (int idx = tid; idx < C * BV; idx += NT) {
      const int i = idx / BV, j = idx % BV;
      float acc = 0.f;
      for (int c = 0; c < D; ++c) acc += s_W[i * D + c] * s_S[c * BV + j];
      s_E[idx] = s_U[idx] - acc;
    }
    __syncthreads();
    // O = Q~ S + A_qk E
    for (int idx = tid; idx < C * BV; idx += NT) {
      const int i = idx / BV, j = idx % BV;
      if (i >= ci.n) continue;
      float acc = 0.f;
      for (int c = 0; c < D; ++c) acc += s_Q[i * D + c] * s_S[c * BV + j];
      for (int m = 0; m <= i; ++m) acc += s_A[i * C + m] * s_E[m * BV + j];
      P.o[((ci.t0 + i) * static_cast<int64_t>(HV) + h) * D + v0 + j] = acc;
    }
    __syncthreads();
    // S = diag(gamma) S + K_end^T E
    for (int idx = tid; idx < D * BV; idx += NT) {
      const int c = idx / BV, j = idx % BV;
      float acc = s_g[c] * s_S[idx];
      for (int i = 0; i < C; ++i) acc += s_K[i * D + c] * s_E[i * BV + j];
      s_S[idx] = acc;
    }
    __syncthreads();
  }
  for (int idx = tid; idx < D * BV; idx += NT) {
    const int c = idx / BV, j = idx % BV;
    if (SBF16)
      static_cast<uint16_t*>(P.pool)[sbase + c * D + v0 + j] = f32_to_bf16_bits(s_S[idx]);
    else
      static_cast<float*>(P.pool)[sbase + c * D + v0 + j] = s_S[idx];
  }
}

template <int D, int C, bool QBF16, bool PERCH, bool SBF16>
static cudaError_t launch_simt_t(const Problem& P, const SimtWorkspace& ws, cudaStream_t st,
                                 const Stages& stages) {
  constexpr int BV = D >= 32 ? 32 : D;
  const int mc = plan_max_chunks(P);
  auto lk = simt_local_kernel<D, C, QBF16, PERCH>;
  constexpr size_t lbytes = SimtLocalSmem<D, C>::bytes;
  cudaError_t e = cudaFuncSetAttribute(lk, cudaFuncAttributeMaxDynamicSharedMemorySize, lbytes);
  if (e != cudaSuccess) return e;
  if (mc > 0) {
    lk<<<dim3(mc, P.HV), 256, lbytes, st>>>(P, ws, ChunkWindow{0, 0}, 0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  stages.mark(2, st);
  auto sk = simt_scan_kernel<D, C, BV, SBF16>;
  constexpr size_t sbytes = SimtScanSmem<D, C, BV>::bytes;
  if ((e = cudaFuncSetAttribute(sk, cudaFuncAttributeMaxDynamicSharedMemorySize, sbytes)) != cudaSuccess)
    return e;
  const unsigned ctas = seq_head_tile_ctas(P, D / BV);
  if (ctas == 0) return cudaErrorInvalidConfiguration;
  sk<<<ctas, 256, sbytes, st>>>(P, ws);
  e = cudaGetLastError();
  stages.mark(3, st);
  return e;
}

template <int D, int C>
static cudaError_t launch_simt_dc(const Problem& P, const SimtWorkspace& ws, bool q, bool pc,
                                  bool sb, cudaStream_t st, const Stages& g) {
  if (q) {
    if (pc) return sb ? launch_simt_t<D, C, true, true, true>(P, ws, st, g)
                      : launch_simt_t<D, C, true, true, false>(P, ws, st, g);
    return sb ? launch_simt_t<D, C, true, false, true>(P, ws, st, g)
              : launch_simt_t<D, C, true, false, false>(P, ws, st, g);
  }
  if (pc) return sb ? launch_simt_t<D, C, false, true, true>(P, ws, st, g)
                    : launch_simt_t<D, C, false, true, false>(P, ws, st, g);
  return sb ? launch_simt_t<D, C, false, false, true>(P, ws, st, g)
            : launch_simt_t<D, C, false, false, false>(P, ws, st, g);
}

template <int D>
static cudaError_t launch_simt_d(const Problem& P, const SimtWorkspace& ws, bool q, bool pc,
                                 bool sb, cudaStream_t st, const Stages& g) {
  switch (P.chunk) {
    case 16: return launch_simt_dc<D, 16>(P, ws, q, pc, sb, st, g);
    case 32: return launch_simt_dc<D, 32>(P, ws, q, pc, sb, st, g);
    default: return launch_simt_dc<D, 64>(P, ws, q, pc, sb, st, g);
  }
}

cudaError_t launch_prefill_simt(const Problem& P, void* workspace, bool qbf16, bool perch,
                                bool sbf16, cudaStream_t stream, const Stages& st) {
  SimtWorkspace ws;
  simt_layout(P, static_cast<char*>(workspace), &ws);
  st.mark(0, stream);
  cudaError_t e = launch_plan(P, ws.plan, stream);
  if (e != cudaSuccess) return e;
  st.mark(1, stream);
  if (P.D == 128) return launch_simt_d<128>(P, ws, qbf16, perch, sbf16, stream, st);
  return launch_simt_d<16>(P, ws, qbf16, perch, sbf16, stream, st);
}

}  // namespace kda
