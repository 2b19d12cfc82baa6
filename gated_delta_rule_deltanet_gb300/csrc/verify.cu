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
// The verify kernel: one CTA per (sequence, value head); warp w owns the value columns
// [CW w, CW w + CW) of the state with all d_k key rows, lane = (row group, column
// quad): RPT consecutive key rows x 4 value columns in registers.  Every sum over key
// channels (the prediction S k^, the read S q^, the norms of k and q) is a sum over the
// lane's rows followed by shuffles between the row-group lanes of its warp: no shared
// memory reduction and no block barrier inside the token loop.
#include <algorithm>

#include "kda_common.cuh"
#include "tc_utils.cuh"


namespace kda {

// polls before a wait on a copy is declared stuck
__host__ __device__ constexpr uint32_t kda_wait_limit() { return 1u << 22; }

template <int D, int NT>
struct VerifyMap {
  static constexpr int NW = NT / 32;     // warps
  static constexpr int CW = D / NW;      // value columns per warp
  static constexpr int NQ = CW / 4;      // column quads per warp
  static constexpr int NG = 32 / NQ;     // row groups per warp
  static constexpr int RPT = D / NG;     // key rows per lane
  static_assert(CW % 4 == 0 && 32 % NQ == 0 && D % NG == 0, "value columns in quads over the warps");
};

// sum over the row-group lanes of a warp (lanes that differ in the bits above the quad bits)
template <int NQ>
__device__ __forceinline__ float rowgroup_sum(float x) {
#pragma unroll
  for (int off = NQ; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// N consecutive q/k/v elements (bf16 or fp32) at p, widened to fp32: 16-byte loads where N
// and the alignment allow (N % 8 for bf16, N % 4 for fp32), else element by element
template <bool BF16, int N>
__device__ __forceinline__ void load_row(const unsigned char* p, float* x) {
  if constexpr (BF16 && N % 8 == 0) {
#pragma unroll
    for (int e = 0; e < N; e += 8) tc::bf16x8_load(p + 2 * e, x + e);
  } else if constexpr (!BF16 && N % 4 == 0) {
#pragma unroll
    for (int e = 0; e < N; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + 4 * e);
      x[e] = v.x; x[e + 1] = v.y; x[e + 2] = v.z; x[e + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e)
      x[e] = BF16 ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(p)[e]) << 16)
                  : reinterpret_cast<const float*>(p)[e];
  }
}

// N consecutive fp32 values to global memory (float4 stores when N % 4 == 0)
template <int N>
__device__ __forceinline__ void store_rows(float* p, const float* x, float scale) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int e = 0; e < N; e += 4)
      *reinterpret_cast<float4*>(p + e) = make_float4(x[e] * scale, x[e + 1] * scale, x[e + 2] * scale,
                                                      x[e + 3] * scale);
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) p[e] = x[e] * scale;
  }
}

// Shared-memory map of the verify kernel: the state buffer (the next pair's state, bulk-copied
// while the current pair is worked on), then two groups of staged token inputs.
template <int D, bool QBF16, bool SBF16, bool PERCH>
struct VerifySmem {
  static constexpr int ES = QBF16 ? 2 : 4;
  static constexpr int TB = 8;                 // tokens per staged group
  static constexpr int GW = PERCH ? D : 4;     // log-decay floats staged per token
  static constexpr int STATE = D * D * (SBF16 ? 2 : 4);
  static constexpr int O_K = 0, O_Q = O_K + TB * D * ES, O_V = O_Q + TB * D * ES;
  static constexpr int O_G = O_V + TB * D * ES, O_B = O_G + TB * GW * 4, BUF = O_B + TB * 4;
  static constexpr int BYTES = STATE + 2 * BUF;
  static_assert(STATE % 16 == 0 && BUF % 16 == 0, "16-byte aligned pieces");
};

// Persistent: each CTA walks the (sequence, value head) pairs blockIdx.x, blockIdx.x + gridDim.x,
// ...  A pair's state arrives in shared memory by one bulk copy issued while the previous pair
// is worked on, and is moved into registers at the pair's start; its window's token inputs
// arrive in groups of TB tokens by cp.async, each group staged while the one before it is
// worked on (the next pair's first group while this pair's last group is).  The token loop
// itself has no barrier and no global load.
// DELTA = false: the additive write (no prediction), a template parameter so that the
// delta rule's code carries no test of it
template <int D, int NT, bool QBF16, bool SBF16, bool PERCH, bool DELTA>
__global__ void __launch_bounds__(NT, 2) verify_window_kernel(Problem P, int window, float* ring,
                                                              int rec, int npairs, int g16) {
  using M = VerifyMap<D, NT>;
  using L = VerifySmem<D, QBF16, SBF16, PERCH>;
  constexpr int RPT = M::RPT, NQ = M::NQ, ES = L::ES, TB = L::TB, GW = L::GW;
  extern __shared__ __align__(128) unsigned char vsmem[];
  __shared__ uint64_t s_sbar;                  // bulk copy of a pair's state
  unsigned char* const sstate = vsmem;
  unsigned char* const sbuf = vsmem + L::STATE;

  const int HV = P.HV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cq = lane % NQ, rg = lane / NQ;
  const int col = warp * M::CW + 4 * cq;       // this lane's 4 value columns
  const int row0 = rg * RPT;                   // and its key rows [row0, row0 + RPT)
  const int ngroups = (window + TB - 1) / TB;

  auto slot_of = [&](int pr) -> uint32_t { return P.slot_idx[pr / HV]; };
  auto valid = [&](int pr) -> bool { return slot_of(pr) < static_cast<uint32_t>(P.num_slots); };
  // one thread: the bulk copy of pair pr's state into the state buffer
  auto copy_state = [&](int pr) {
    const int64_t base = (static_cast<int64_t>(slot_of(pr)) * HV + pr % HV) * D * D;
    tc::mbar_arrive_expect_tx(&s_sbar, L::STATE);
    tc::bulk_load(tc::smem_u32(sstate), static_cast<const char*>(P.pool) + base * (SBF16 ? 2 : 4),
                  L::STATE, &s_sbar);
  };
  // cp.async copies of tokens [TB gi, TB gi + TB) of pair pr's window into group buffer bi
  auto stage = [&](int pr, int gi, int bi) {
    const int b = pr / HV, h = pr % HV, kh = h / (HV / P.HK);
    const uint32_t sb = tc::smem_u32(sbuf + bi * L::BUF);
    const int t0 = TB * gi, nt = min(TB, window - t0);
    constexpr int PR = D * ES / 16;            // 16-byte pieces of a k, q or v row
    for (int u = tid; u < nt * PR; u += NT) {
      const int t = u / PR, pc = u % PR;
      const int64_t row_t = static_cast<int64_t>(b) * window + t0 + t;
      const char* kp = static_cast<const char*>(P.k) + (row_t * P.k_stride + static_cast<int64_t>(kh) * D) * ES;
      const char* qp = static_cast<const char*>(P.q) + (row_t * P.q_stride + static_cast<int64_t>(kh) * D) * ES;
      const char* vp = static_cast<const char*>(P.v) + (row_t * P.v_stride + static_cast<int64_t>(h) * D) * ES;
      tc::cp_async16(sb + L::O_K + (t * D * ES) + 16 * pc, kp + 16 * pc, 16u);
      tc::cp_async16(sb + L::O_Q + (t * D * ES) + 16 * pc, qp + 16 * pc, 16u);
      tc::cp_async16(sb + L::O_V + (t * D * ES) + 16 * pc, vp + 16 * pc, 16u);
    }
    if constexpr (PERCH) {
      if (g16) {                               // 16-byte pieces where the log-decay array allows
        for (int u = tid; u < nt * (D / 4); u += NT) {
          const int t = u / (D / 4), pc = u % (D / 4);
          const int64_t row_t = static_cast<int64_t>(b) * window + t0 + t;
          tc::cp_async16(sb + L::O_G + t * GW * 4 + 16 * pc, P.g + (row_t * HV + h) * D + 4 * pc, 16u);
        }
      } else {                                 // the entry point asks for 4-byte alignment only
        for (int u = tid; u < nt * D; u += NT) {
          const int t = u / D, c = u % D;
          const int64_t row_t = static_cast<int64_t>(b) * window + t0 + t;
          tc::cp_async4(sb + L::O_G + (t * GW + c) * 4, P.g + (row_t * HV + h) * D + c, 4u);
        }
      }
    }
    if (tid < nt) {
      const int64_t row_t = static_cast<int64_t>(b) * window + t0 + tid;
      if (!PERCH) tc::cp_async4(sb + L::O_G + tid * GW * 4, P.g + row_t * HV + h, 4u);
      tc::cp_async4(sb + L::O_B + tid * 4, P.beta + row_t * HV + h, 4u);
    }
    tc::cp_async_commit();
  };

  const int p0 = blockIdx.x;
  if (tid == 0) {
    tc::mbar_init(&s_sbar, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0 && valid(p0)) copy_state(p0);
  stage(p0, 0, 0);
  uint32_t sphase = 0;                         // state copies waited for
  int gcount = 0;                              // token groups consumed (buffer gcount % 2)
  bool abort = false;
  for (int pr = p0; pr < npairs && !abort; pr += gridDim.x) {
    const int b = pr / HV, h = pr % HV;
    const bool ok_slot = valid(pr);            // block-uniform
    const int pn = pr + gridDim.x;
    float2 S01[RPT], S23[RPT];                 // the lane's state: columns (0, 1) and (2, 3)
    if (ok_slot) {
      const bool got = tc::mbar_wait_bounded(&s_sbar, sphase & 1, kda_wait_limit());
      if (__syncthreads_or(!got)) {            // sphase still names the copy in flight
        if (tid == 0) raise_device_error(P.err, KDA_DEVERR_TIMEOUT);
        abort = true;
        break;
      }
      ++sphase;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float4 v = load4<SBF16>(sstate, static_cast<int64_t>(row0 + i) * D + col);
        S01[i] = make_float2(v.x, v.y);
        S23[i] = make_float2(v.z, v.w);
      }
    } else if (tid == 0) {
      raise_device_error(P.err, KDA_DEVERR_SLOT_RANGE);
    }
    __syncthreads();                           // the state buffer has been read
    if (tid == 0 && pn < npairs && valid(pn)) {
      tc::fence_async_smem();
      copy_state(pn);
    }
    for (int gi = 0; gi < ngroups; ++gi, ++gcount) {
      unsigned char* buf = sbuf + (gcount & 1) * L::BUF;
      const int nt = min(TB, window - TB * gi);
      tc::cp_async_wait_all();
      __syncthreads();                         // this group staged; the other buffer free
      if (gi + 1 < ngroups) stage(pr, gi + 1, (gcount + 1) & 1);
      else if (pn < npairs) stage(pn, 0, (gcount + 1) & 1);
      // the group's decays alpha = exp(g), once per value (every lane reads its rows' alphas)
      for (int u = tid; u < nt * (PERCH ? D : 1); u += NT) {
        float* gp = reinterpret_cast<float*>(buf + L::O_G) + (PERCH ? u : u * GW);
        *gp = __expf(*gp);
      }
      __syncthreads();
      if (!ok_slot) continue;
      for (int t = 0; t < nt; ++t) {
        const int64_t row_t = static_cast<int64_t>(b) * window + TB * gi + t;
        float kr[RPT], a[RPT];
        load_row<QBF16, RPT>(buf + L::O_K + (t * D + row0) * ES, kr);
        if constexpr (PERCH) {
          load_row<false, RPT>(buf + L::O_G + (t * GW + row0) * 4, a);
        } else {
          const float a0 = *reinterpret_cast<const float*>(buf + L::O_G + t * GW * 4);
#pragma unroll
          for (int i = 0; i < RPT; ++i) a[i] = a0;
        }
        float* rec_p = ring + (row_t * HV + h) * rec;   // the record of this token: [k^ | e | alpha]
        if (warp == 0 && cq == 0) {
          if (PERCH) store_rows<RPT>(rec_p + 2 * D + row0, a, 1.f);
          else if (rg == 0) rec_p[2 * D] = a[0];
        }
        // forget and predict (raw k; its norm applies after the sum, which is linear); the
        // state's 4 columns as two pairs, two-wide arithmetic
        float2 p01 = make_float2(0.f, 0.f), p23 = make_float2(0.f, 0.f);
        float ssk = 0.f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const float2 ai = make_float2(a[i], a[i]), ki = make_float2(kr[i], kr[i]);
          S01[i] = mul2(S01[i], ai);
          S23[i] = mul2(S23[i], ai);
          if constexpr (DELTA) {
            p01 = fma2(S01[i], ki, p01);
            p23 = fma2(S23[i], ki, p23);
          }
          ssk += kr[i] * kr[i];
        }
        ssk = rowgroup_sum<NQ>(ssk);
        const float kscale = P.l2norm ? rsqrtf(ssk + 1e-6f) : 1.f;
        float4 vhat = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (DELTA) {
          vhat.x = rowgroup_sum<NQ>(p01.x) * kscale; vhat.y = rowgroup_sum<NQ>(p01.y) * kscale;
          vhat.z = rowgroup_sum<NQ>(p23.x) * kscale; vhat.w = rowgroup_sum<NQ>(p23.y) * kscale;
        }
        float vv[4];
        load_row<QBF16, 4>(buf + L::O_V + (t * D + col) * ES, vv);
        const float beta = *reinterpret_cast<const float*>(buf + L::O_B + 4 * t);
        const float4 e = make_float4(beta * (vv[0] - vhat.x), beta * (vv[1] - vhat.y),
                                     beta * (vv[2] - vhat.z), beta * (vv[3] - vhat.w));
        const float2 e01 = make_float2(e.x, e.y), e23 = make_float2(e.z, e.w);
        // write and read (k reloaded from shared memory rather than kept across the sums)
        float qr[RPT];
        load_row<QBF16, RPT>(buf + L::O_Q + (t * D + row0) * ES, qr);
        load_row<QBF16, RPT>(buf + L::O_K + (t * D + row0) * ES, kr);
        float2 o01 = make_float2(0.f, 0.f), o23 = make_float2(0.f, 0.f);
        float ssq = 0.f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const float2 kc = make_float2(kr[i] * kscale, kr[i] * kscale), qi = make_float2(qr[i], qr[i]);
          S01[i] = fma2(kc, e01, S01[i]);
          S23[i] = fma2(kc, e23, S23[i]);
          o01 = fma2(S01[i], qi, o01);
          o23 = fma2(S23[i], qi, o23);
          ssq += qr[i] * qr[i];
        }
        ssq = rowgroup_sum<NQ>(ssq);
        const float qscale = (P.l2norm ? rsqrtf(ssq + 1e-6f) : 1.f) * P.scale;
        float4 o;
        o.x = rowgroup_sum<NQ>(o01.x) * qscale; o.y = rowgroup_sum<NQ>(o01.y) * qscale;
        o.z = rowgroup_sum<NQ>(o23.x) * qscale; o.w = rowgroup_sum<NQ>(o23.y) * qscale;
        // k^ and e into the record, and the output
        if (warp == 0 && cq == 0) store_rows<RPT>(rec_p + row0, kr, kscale);
        if (rg == 0) {
          *reinterpret_cast<float4*>(rec_p + D + col) = e;
          *reinterpret_cast<float4*>(P.o + (row_t * HV + h) * D + col) = o;
        }
      }
    }
  }
  // nothing may still be landing in shared memory when the CTA exits: the last staged token
  // group, and (after an abort) a state copy in flight
  tc::cp_async_wait_all();
  if (abort && tid == 0) tc::mbar_wait_bounded(&s_sbar, sphase & 1, kda_wait_limit());
}

// The fold keeps the decode step's layout: thread = 16-byte column group of several state
// rows; k^ and alpha of each record pass through shared memory (one or two barriers per
// accepted record, few per sequence).
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

// SMs of the current device (cached per device)
template <int D, int NT, bool Q, bool SB, bool PC>
static cudaError_t launch_verify_t(const Problem& P, int window, float* ring, cudaStream_t s) {
  const int64_t pairs = static_cast<int64_t>(P.num_seqs) * P.HV;
  // two resident CTAs per SM walk the pairs
  const int grid = static_cast<int>(std::min<int64_t>(pairs, 2 * static_cast<int64_t>(sm_count())));
  constexpr int bytes = VerifySmem<D, Q, SB, PC>::BYTES;
  auto k = (P.flags & KDA_FLAG_NO_DELTA) ? verify_window_kernel<D, NT, Q, SB, PC, false>
                                         : verify_window_kernel<D, NT, Q, SB, PC, true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  const bool g16 = (reinterpret_cast<uintptr_t>(P.g) & 15u) == 0;
  k<<<dim3(static_cast<unsigned>(grid)), NT, bytes, s>>>(P, window, ring, ring_record_elems(D, PC),
                                                          static_cast<int>(pairs), g16 ? 1 : 0);
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
