// verify.cu -- speculative-decode verification window and the fold of accepted records.
//
// Modular MAX "gated_delta" module: the verify kernel runs the gated delta
// recurrence over a window of draft tokens and records a ring instead of
// writing the state back; the fold applies the accepted prefix of those records
// to the state pool.  A record holds what one token's update needs
// (k^, the corrected value e, the decay alpha), so the fold replays the forget
// and write steps of the KDA update ("You Could Have Come Up With Kimi Delta
// Attention", sec. 4) exactly: S <- S Diag(alpha) + e k^T.
//
// Both kernels use the decode step's layout: one CTA per (sequence, value head),
// each thread holding 16-byte column groups of several state rows in registers,
// reductions over key channels by warp shuffles plus one shared-memory combine.
#include "kda_common.cuh"

namespace kda {

// DELTA = false: the additive write (no prediction), a template parameter so that the
// delta rule's code carries no test of it
template <int D, int NT, bool QBF16, bool SBF16, bool PERCH, bool DELTA>
__global__ void __launch_bounds__(NT) verify_window_kernel(Problem P, int window, float* ring,
                                                           int rec) {
  constexpr int VEC = 4;
  constexpr int TPR = D / VEC;
  constexpr int RPP = NT / TPR;
  constexpr int RPT = D / RPP;
  constexpr int NWARP = NT / 32;
  // token inputs double-buffered: token t + 1's are written while token t is worked on and
  // published by token t's second reduction, so a token costs two barriers (its reductions)
  __shared__ float s_k[2][D], s_q[2][D], s_a[2][D];
  __shared__ float s_red[2][NWARP][D];
  __shared__ float s_scale[2][2];
  static_assert(NT >= D, "one key channel per thread");

  const int HV = P.HV;
  const int64_t bh = blockIdx.x;
  const int b = static_cast<int>(bh / HV), h = static_cast<int>(bh % HV);
  const int kh = h / (HV / P.HK);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cg = tid % TPR, r0 = tid / TPR;

  const uint32_t slot = P.slot_idx[b];
  if (slot >= static_cast<uint32_t>(P.num_slots)) {
    if (tid == 0) raise_device_error(P.err, KDA_DEVERR_SLOT_RANGE);
    return;
  }
  const int64_t state_base = (static_cast<int64_t>(slot) * HV + h) * D * D;
  float4 S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    S[i] = load4<SBF16>(P.pool, state_base + static_cast<int64_t>(r0 + i * RPP) * D + cg * VEC);

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

  auto stage = [&](int t) {                     // token t's k, q, alpha into buffer t & 1
    const int64_t row_t = static_cast<int64_t>(b) * window + t;
    if (tid < D) {
      const int bt = t & 1;
      s_k[bt][tid] = load_elem<QBF16>(P.k, row_t * P.k_stride + static_cast<int64_t>(kh) * D + tid);
      s_q[bt][tid] = load_elem<QBF16>(P.q, row_t * P.q_stride + static_cast<int64_t>(kh) * D + tid);
      s_a[bt][tid] = expf(PERCH ? P.g[(row_t * HV + h) * D + tid] : P.g[row_t * HV + h]);
    }
  };
  stage(0);
  __syncthreads();
  for (int t = 0; t < window; ++t) {
    const int64_t row_t = static_cast<int64_t>(b) * window + t;
    const int bt = t & 1;
    const float* sk = s_k[bt];
    const float* sq = s_q[bt];
    const float* sa = s_a[bt];
    // the L2 norms of k and q (warps 0 and 1), published by the first reduction below: the
    // products before it use the raw k and q and take the scales afterwards (they are linear)
    if (warp < 2) {
      constexpr int kStep = NWARP > 1 ? 2 : 1;
      for (int which = NWARP > 1 ? warp : 0; which < 2; which += kStep) {
        const float* x = which == 0 ? sk : sq;
        float ss = 0.f;
        for (int c = lane; c < D; c += 32) ss += x[c] * x[c];
        ss = warp_sum(ss);
        if (lane == 0) {
          const float inv = P.l2norm ? rsqrtf(ss + 1e-6f) : 1.f;
          s_scale[bt][which] = which == 0 ? inv : inv * P.scale;
        }
      }
    }
    const float vbeta = P.beta[row_t * HV + h];
    const float4 vv = load4<QBF16>(P.v, row_t * P.v_stride + static_cast<int64_t>(h) * D + cg * VEC);

    float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = r0 + i * RPP;
      const float a = sa[r], kr = sk[r];
      S[i].x *= a; S[i].y *= a; S[i].z *= a; S[i].w *= a;
      part.x += S[i].x * kr; part.y += S[i].y * kr; part.z += S[i].z * kr; part.w += S[i].w * kr;
    }
    // additive write (no delta rule): nothing is predicted, e = beta v
    float4 vhat = make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (DELTA) vhat = reduce_rows(part, 0);
    else __syncthreads();
    const float kscale = s_scale[bt][0], qscale = s_scale[bt][1];
    vhat.x *= kscale; vhat.y *= kscale; vhat.z *= kscale; vhat.w *= kscale;
    const float4 e = make_float4(vbeta * (vv.x - vhat.x), vbeta * (vv.y - vhat.y),
                                 vbeta * (vv.z - vhat.z), vbeta * (vv.w - vhat.w));
    float4 opart = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = r0 + i * RPP;
      const float kc = sk[r] * kscale, qr = sq[r];
      S[i].x += kc * e.x; S[i].y += kc * e.y; S[i].z += kc * e.z; S[i].w += kc * e.w;
      opart.x += S[i].x * qr; opart.y += S[i].y * qr; opart.z += S[i].z * qr; opart.w += S[i].w * qr;
    }
    // the record of this token: [k^ | e | alpha]
    float* rec_p = ring + (row_t * HV + h) * rec;
    if (tid < D) {
      rec_p[tid] = sk[tid] * kscale;
      if (PERCH) rec_p[2 * D + tid] = sa[tid];
    }
    if (!PERCH && tid == 0) rec_p[2 * D] = sa[0];
    if (r0 == 0) *reinterpret_cast<float4*>(rec_p + D + cg * VEC) = e;
    // the next token into the other buffer (last read before this token's first barrier)
    if (t + 1 < window) stage(t + 1);
    float4 o = reduce_rows(opart, 1);
    o.x *= qscale; o.y *= qscale; o.z *= qscale; o.w *= qscale;
    if (r0 == 0) *reinterpret_cast<float4*>(P.o + (row_t * HV + h) * D + cg * VEC) = o;
  }
}

template <int D, int NT, bool SBF16, bool PERCH>
__global__ void __launch_bounds__(NT) fold_accepted_kernel(Problem P, int window, const float* ring,
                                                           int rec, const uint32_t* accepted) {
  constexpr int VEC = 4;
  constexpr int TPR = D / VEC;
  constexpr int RPP = NT / TPR;
  constexpr int RPT = D / RPP;
  __shared__ float s_k[D], s_a[D];

  const int HV = P.HV;
  const int64_t bh = blockIdx.x;
  const int b = static_cast<int>(bh / HV), h = static_cast<int>(bh % HV);
  const int tid = threadIdx.x, cg = tid % TPR, r0 = tid / TPR;
  const uint32_t slot = P.slot_idx[b];
  const uint32_t acc = accepted[b];
  if (slot >= static_cast<uint32_t>(P.num_slots) || acc > static_cast<uint32_t>(window)) {
    if (tid == 0)
      raise_device_error(P.err, slot >= static_cast<uint32_t>(P.num_slots) ? KDA_DEVERR_SLOT_RANGE
                                                                           : KDA_DEVERR_ACCEPTED);
    return;
  }
  if (acc == 0) return;
  const int64_t state_base = (static_cast<int64_t>(slot) * HV + h) * D * D;
  float4 S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    S[i] = load4<SBF16>(P.pool, state_base + static_cast<int64_t>(r0 + i * RPP) * D + cg * VEC);
  // the next record, loaded into registers while the current one is applied
  static_assert(NT >= D, "one key channel per thread");
  float nk = 0.f, na = 0.f;
  float4 ne;
  auto fetch = [&](uint32_t t) {
    const float* rec_p = ring + ((static_cast<int64_t>(b) * window + t) * HV + h) * rec;
    if (tid < D) {
      nk = rec_p[tid];
      na = PERCH ? rec_p[2 * D + tid] : rec_p[2 * D];
    }
    ne = *reinterpret_cast<const float4*>(rec_p + D + cg * VEC);
  };
  fetch(0);
  for (uint32_t t = 0; t < acc; ++t) {
    __syncthreads();
    if (tid < D) {
      s_k[tid] = nk;
      s_a[tid] = na;
    }
    const float4 e = ne;
    if (t + 1 < acc) fetch(t + 1);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = r0 + i * RPP;
      const float a = s_a[r], kc = s_k[r];
      S[i].x = a * S[i].x + kc * e.x;
      S[i].y = a * S[i].y + kc * e.y;
      S[i].z = a * S[i].z + kc * e.z;
      S[i].w = a * S[i].w + kc * e.w;
    }
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    store4<SBF16>(P.pool, state_base + static_cast<int64_t>(r0 + i * RPP) * D + cg * VEC, S[i]);
}

// [k^ (D) | e (D) | alpha (D per channel, or 1 padded to 4 so records stay 16-byte aligned)]
int ring_record_elems(int D, bool perch) { return D + D + (perch ? D : 4); }

template <int D, int NT, bool Q, bool SB, bool PC>
static cudaError_t launch_verify_t(const Problem& P, int window, float* ring, cudaStream_t s) {
  const int64_t blocks = static_cast<int64_t>(P.num_seqs) * P.HV;
  if (P.flags & KDA_FLAG_NO_DELTA)
    verify_window_kernel<D, NT, Q, SB, PC, false><<<dim3(static_cast<unsigned>(blocks)), NT, 0, s>>>(
        P, window, ring, ring_record_elems(D, PC));
  else
    verify_window_kernel<D, NT, Q, SB, PC, true><<<dim3(static_cast<unsigned>(blocks)), NT, 0, s>>>(
        P, window, ring, ring_record_elems(D, PC));
  return cudaGetLastError();
}

template <int D, int NT>
static cudaError_t launch_verify_d(const Problem& P, int window, float* ring, bool q, bool sb,
                                   bool pc, cudaStream_t s) {
  if (q) {
    if (sb) return pc ? launch_verify_t<D, NT, true, true, true>(P, window, ring, s)
                      : launch_verify_t<D, NT, true, true, false>(P, window, ring, s);
    return pc ? launch_verify_t<D, NT, true, false, true>(P, window, ring, s)
              : launch_verify_t<D, NT, true, false, false>(P, window, ring, s);
  }
  if (sb) return pc ? launch_verify_t<D, NT, false, true, true>(P, window, ring, s)
                    : launch_verify_t<D, NT, false, true, false>(P, window, ring, s);
  return pc ? launch_verify_t<D, NT, false, false, true>(P, window, ring, s)
            : launch_verify_t<D, NT, false, false, false>(P, window, ring, s);
}

cudaError_t launch_verify(const Problem& P, int window, float* ring, bool qbf16, bool sbf16,
                          bool perch, cudaStream_t stream) {
  if (P.D == 128) return launch_verify_d<128, 256>(P, window, ring, qbf16, sbf16, perch, stream);
  return launch_verify_d<16, 32>(P, window, ring, qbf16, sbf16, perch, stream);
}

template <int D, int NT, bool SB, bool PC>
static cudaError_t launch_fold_t(const Problem& P, int window, const float* ring,
                                 const uint32_t* accepted, cudaStream_t s) {
  const int64_t blocks = static_cast<int64_t>(P.num_seqs) * P.HV;
  fold_accepted_kernel<D, NT, SB, PC><<<dim3(static_cast<unsigned>(blocks)), NT, 0, s>>>(
      P, window, ring, ring_record_elems(D, PC), accepted);
  return cudaGetLastError();
}

cudaError_t launch_fold(const Problem& P, int window, const float* ring, const uint32_t* accepted,
                        bool sbf16, bool perch, cudaStream_t s) {
  if (P.D == 128) {
    if (sbf16) return perch ? launch_fold_t<128, 256, true, true>(P, window, ring, accepted, s)
                            : launch_fold_t<128, 256, true, false>(P, window, ring, accepted, s);
    return perch ? launch_fold_t<128, 256, false, true>(P, window, ring, accepted, s)
                 : launch_fold_t<128, 256, false, false>(P, window, ring, accepted, s);
  }
  if (sbf16) return perch ? launch_fold_t<16, 32, true, true>(P, window, ring, accepted, s)
                          : launch_fold_t<16, 32, true, false>(P, window, ring, accepted, s);
  return perch ? launch_fold_t<16, 32, false, true>(P, window, ring, accepted, s)
               : launch_fold_t<16, 32, false, false>(P, window, ring, accepted, s);
}

}  // namespace kda
