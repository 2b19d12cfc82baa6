// decode.cu -- one recurrent decode step of the gated delta rule.
//
// "You Could Have Come Up With Kimi Delta Attention", sec. 5 (fused recurrent
// kernel: decay, predict, correct, write, read on a state tile that one program
// owns) and the Modular MAX "gated_delta" module (five per-token steps, GQA key
// head = value head // ratio, slot-indexed pool updated in place).
//
// The step is bound by HBM: every (sequence, value head) reads and writes its
// d_k x d_v state once and touches only a few hundred bytes of token data.
// One CTA owns one (sequence, value head) state.  Its threads tile the state
// as rows (key channels) x 4-column groups so that every load and store is a
// 16-byte vector of consecutive value columns and each warp moves whole
// 512-byte rows.  All state loads are issued before the token data is
// reduced, so one CTA keeps its whole state in flight; the two reductions over
// key channels (predict and read) are warp shuffles plus one shared-memory
// combine across warps.
#include "kda_common.cuh"

namespace kda {

// DELTA = false: the additive write (no prediction), a template parameter so that the
// delta rule's code carries no test of it
template <int D, int NT, bool QBF16, bool SBF16, bool PERCH, bool DELTA>
__global__ void __launch_bounds__(NT) decode_step_kernel(Problem P) {
  constexpr int VEC = 4;
  constexpr int TPR = D / VEC;        // threads across one state row
  static_assert(TPR >= 1 && TPR <= 32 && 32 % TPR == 0, "row must tile a warp");
  constexpr int RPP = NT / TPR;       // rows covered by one pass of the CTA
  static_assert(D % RPP == 0, "rows must tile");
  constexpr int RPT = D / RPP;        // rows held by each thread
  constexpr int NWARP = NT / 32;

  __shared__ float s_k[D], s_q[D], s_a[D];
  __shared__ float s_red[2][NWARP][D];
  __shared__ float s_scale[2];

  const int HV = P.HV;
  const int64_t bh = blockIdx.x;
  const int b = static_cast<int>(bh / HV);
  const int h = static_cast<int>(bh % HV);
  const int kh = h / (HV / P.HK);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int cg = tid % TPR;
  const int r0 = tid / TPR;

  const uint32_t slot = P.slot_idx[b];
  if (slot >= static_cast<uint32_t>(P.num_slots)) {
    if (tid == 0) raise_device_error(P.err, KDA_DEVERR_SLOT_RANGE);
    return;
  }
  const int64_t state_base = (static_cast<int64_t>(slot) * HV + h) * D * D;

  // 1. issue the state loads first
  float4 S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = r0 + i * RPP;
    S[i] = load4<SBF16>(P.pool, state_base + static_cast<int64_t>(row) * D + cg * VEC);
  }

  // 2. token data: k, q (key head), log-decay, then the L2 norms
  const int64_t qrow = static_cast<int64_t>(b) * P.q_stride + static_cast<int64_t>(kh) * D;
  const int64_t krow = static_cast<int64_t>(b) * P.k_stride + static_cast<int64_t>(kh) * D;
  for (int c = tid; c < D; c += NT) {
    s_k[c] = load_elem<QBF16>(P.k, krow + c);
    s_q[c] = load_elem<QBF16>(P.q, qrow + c);
    const float gc = PERCH ? P.g[(static_cast<int64_t>(b) * HV + h) * D + c]
                           : P.g[static_cast<int64_t>(b) * HV + h];
    s_a[c] = expf(gc);
  }
  __syncthreads();
  if (warp < 2) {
    // warp 0 reduces |k|^2 and warp 1 |q|^2 (a single-warp CTA does both)
    constexpr int kStep = NWARP > 1 ? 2 : 1;
    for (int which = NWARP > 1 ? warp : 0; which < 2; which += kStep) {
      const float* x = which == 0 ? s_k : s_q;
      float ss = 0.f;
      for (int c = lane; c < D; c += 32) ss += x[c] * x[c];
      ss = warp_sum(ss);
      if (lane == 0) {
        const float inv = P.l2norm ? rsqrtf(ss + 1e-6f) : 1.f;
        s_scale[which] = which == 0 ? inv : inv * P.scale;
      }
    }
  }
  __syncthreads();
  const float kscale = s_scale[0], qscale = s_scale[1];

  const float vbeta = P.beta[static_cast<int64_t>(b) * HV + h];
  const float4 vv = load4<QBF16>(P.v, static_cast<int64_t>(b) * P.v_stride +
                                          static_cast<int64_t>(h) * D + cg * VEC);

  // 3. forget, then partial predictions over this thread's rows
  float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = r0 + i * RPP;
    const float a = s_a[row];
    const float kc = s_k[row] * kscale;
    S[i].x *= a; S[i].y *= a; S[i].z *= a; S[i].w *= a;
    part.x += S[i].x * kc; part.y += S[i].y * kc; part.z += S[i].z * kc; part.w += S[i].w * kc;
  }
  auto reduce_rows = [&](float4 p, int buf) -> float4 {
#pragma unroll
    for (int off = TPR; off < 32; off <<= 1) {
      p.x += __shfl_xor_sync(0xffffffffu, p.x, off);
      p.y += __shfl_xor_sync(0xffffffffu, p.y, off);
      p.z += __shfl_xor_sync(0xffffffffu, p.z, off);
      p.w += __shfl_xor_sync(0xffffffffu, p.w, off);
    }
    if (lane < TPR) *reinterpret_cast<float4*>(&s_red[buf][warp][cg * VEC]) = p;
    __syncthreads();
    float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NWARP; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(&s_red[buf][w][cg * VEC]);
      tot.x += x.x; tot.y += x.y; tot.z += x.z; tot.w += x.w;
    }
    return tot;
  };
  // additive write (no delta rule): nothing is predicted, e = beta v
  float4 vhat = make_float4(0.f, 0.f, 0.f, 0.f);
  if constexpr (DELTA) vhat = reduce_rows(part, 0);

  // 4. correct and write
  const float4 e = make_float4(vbeta * (vv.x - vhat.x), vbeta * (vv.y - vhat.y),
                               vbeta * (vv.z - vhat.z), vbeta * (vv.w - vhat.w));
  float4 opart = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = r0 + i * RPP;
    const float kc = s_k[row] * kscale;
    const float qc = s_q[row] * qscale;
    S[i].x += kc * e.x; S[i].y += kc * e.y; S[i].z += kc * e.z; S[i].w += kc * e.w;
    opart.x += S[i].x * qc; opart.y += S[i].y * qc; opart.z += S[i].z * qc; opart.w += S[i].w * qc;
  }
  // 5. store the state while the read is reduced
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = r0 + i * RPP;
    store4<SBF16>(P.pool, state_base + static_cast<int64_t>(row) * D + cg * VEC, S[i]);
  }
  const float4 o = reduce_rows(opart, 1);
  if (r0 == 0) {
    *reinterpret_cast<float4*>(P.o + (static_cast<int64_t>(b) * HV + h) * D + cg * VEC) = o;
  }
}

template <int D, int NT, bool QBF16, bool SBF16, bool PERCH>
static cudaError_t launch_decode_t(const Problem& P, cudaStream_t stream, const Stages& st) {
  const int64_t blocks = static_cast<int64_t>(P.num_seqs) * P.HV;
  st.mark(0, stream);
  if (P.flags & KDA_FLAG_NO_DELTA)
    decode_step_kernel<D, NT, QBF16, SBF16, PERCH, false><<<dim3(static_cast<unsigned>(blocks)), NT, 0, stream>>>(P);
  else
    decode_step_kernel<D, NT, QBF16, SBF16, PERCH, true><<<dim3(static_cast<unsigned>(blocks)), NT, 0, stream>>>(P);
  cudaError_t e = cudaGetLastError();
  st.mark(1, stream);
  return e;
}

template <int D, int NT>
static cudaError_t launch_decode_d(const Problem& P, bool qbf16, bool sbf16, bool perch,
                                   cudaStream_t s, const Stages& g) {
  if (qbf16) {
    if (sbf16) return perch ? launch_decode_t<D, NT, true, true, true>(P, s, g)
                            : launch_decode_t<D, NT, true, true, false>(P, s, g);
    return perch ? launch_decode_t<D, NT, true, false, true>(P, s, g)
                 : launch_decode_t<D, NT, true, false, false>(P, s, g);
  }
  if (sbf16) return perch ? launch_decode_t<D, NT, false, true, true>(P, s, g)
                          : launch_decode_t<D, NT, false, true, false>(P, s, g);
  return perch ? launch_decode_t<D, NT, false, false, true>(P, s, g)
               : launch_decode_t<D, NT, false, false, false>(P, s, g);
}

cudaError_t launch_decode(const Problem& P, bool qbf16, bool sbf16, bool perch,
                          cudaStream_t stream, const Stages& st) {
  if (P.D == 128) return launch_decode_d<128, 256>(P, qbf16, sbf16, perch, stream, st);
  return launch_decode_d<16, 32>(P, qbf16, sbf16, perch, stream, st);
}

}  // namespace kda
