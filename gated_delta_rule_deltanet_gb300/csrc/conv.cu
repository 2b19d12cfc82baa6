// conv.cu -- the front end before the recurrence: short causal convolution + SiLU over the
// packed [Q | K | V] projection with a slot-indexed conv state, and the gate activations.
//
// The Modular "gated_delta" module names this step (its "Pass 1": the convolution output with
// channels [Q | K | V], a decay with the softplus applied and a beta with the sigmoid applied);
// "From Attention to Learned Memory", sec. 1 applies SiLU to the features; the linear-attention
// page's Mamba-2 section builds the decay from a log-rate and a softplus step.  Per channel c
// and token t of a sequence starting at bos:
//
//     y[t, c] = SiLU(bias[c] + sum_{i < W} w[c, i] x[t - W + 1 + i, c])
//
// with x before bos taken from the sequence's slot of the conv-state pool (the sequence's
// previous W - 1 inputs, oldest first); afterwards the slot holds the last W - 1 inputs.
// The gates: beta = sigmoid(b), log-decay = -exp(A_log[h]) softplus(a + dt_bias).
//
// Bound by HBM: every input element is read once (plus W - 1 rows per 64-token run) and every
// output written once.  A thread owns 8 consecutive channels (16-byte vectors) over a run of
// 64 tokens, keeping the W - 1 previous inputs in registers; consecutive threads take
// consecutive channel groups of the same tokens, so every row is read and written coalesced.
#include <algorithm>

#include "kda_common.cuh"

namespace kda {

struct ConvArgs {
  const void* x;             // [T, CD]
  const float* w;            // [CD, W]
  const float* bias;         // [CD] or null
  const float* a;            // [T, HV * GW]
  const float* b;            // [T, HV]
  const float* A_log;        // [HV] or null
  const float* dt_bias;      // [HV * GW] or null
  const uint32_t* offsets;   // [B + 1], or null: token s is sequence s
  const uint32_t* slot_idx;  // [B] (needed with a conv state)
  void* state;               // [num_slots, CD, W - 1] or null
  void* y;                   // [T, CD]
  float* g;                  // [T, HV * GW]
  float* beta;               // [T, HV]
  int64_t T;
  int32_t B, CD, HV, GW, num_slots;
  int32_t* err;
};

constexpr int kConvRun = 64;          // tokens of one run

__device__ __forceinline__ void tc_cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// x is only read during a call: read-only loads, free to move ahead of the stores of y
template <bool BF16>
__device__ __forceinline__ void ld8(const void* base, int64_t i, float (&x)[8]) {
  if constexpr (BF16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + i));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  } else {
    const float4 p = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
    const float4 q = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i + 4));
    x[0] = p.x; x[1] = p.y; x[2] = p.z; x[3] = p.w; x[4] = q.x; x[5] = q.y; x[6] = q.z; x[7] = q.w;
  }
}

template <bool BF16>
__device__ __forceinline__ void st8(void* base, int64_t i, const float (&x)[8]) {
  if constexpr (BF16) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)             // round to nearest even, two per instruction
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[e]) : "f"(x[2 * e + 1]), "f"(x[2 * e]));
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + i) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(base) + i) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(static_cast<float*>(base) + i + 4) = make_float4(x[4], x[5], x[6], x[7]);
  }
}

template <bool BF16>
__device__ __forceinline__ float ld1(const void* base, int64_t i) {
  if constexpr (BF16) return bf16_bits_to_f32(static_cast<const uint16_t*>(base)[i]);
  else return static_cast<const float*>(base)[i];
}

// SiLU(z) = z sigmoid(z).  For a bf16 result sigmoid(z) = (1 + tanh(z / 2)) / 2 with the
// hardware tanh (one special-function op, absolute error ~2^-11, well inside the bf16
// rounding of the result); for fp32 the exponential and a reciprocal (~2 ulp each).
template <bool BF16>
__device__ __forceinline__ float silu(float z) {
  if constexpr (BF16) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return z * fmaf(0.5f, t, 0.5f);
  } else {
    return z * __fdividef(1.f, 1.f + __expf(-z));   // 0 for z -> -inf
  }
}

// the sequence holding token t: offsets[s] <= t < offsets[s + 1] (empty sequences skipped)
__device__ __forceinline__ int seq_of(const uint32_t* offsets, int B, int64_t t) {
  if (!offsets) return static_cast<int>(t);
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(offsets[mid]) <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// the W - 1 inputs before token t of the sequence starting at bos: rows of x from bos on,
// the slot's conv state before it (zeros without a state or for a slot out of range)
template <bool BF16, int W>
__device__ __forceinline__ void fill_window(const ConvArgs& A, int s, int64_t bos, int64_t t, int c,
                                            float (&win)[W > 1 ? W - 1 : 1][8]) {
  uint32_t slot = 0;
  bool has_state = false;
  if (A.state && W > 1) {
    slot = A.slot_idx[s];
    has_state = slot < static_cast<uint32_t>(A.num_slots);
    if (!has_state) raise_device_error(A.err, KDA_DEVERR_SLOT_RANGE);
  }
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    const int64_t pos = t - (W - 1) + j;
    const int64_t back = bos - pos;             // 1 .. W - 1 before the sequence's start
    if (pos >= bos) {
      ld8<BF16>(A.x, pos * A.CD + c, win[j]);
    } else if (has_state && back <= W - 1) {    // (more only with offsets out of order)
      const int idx = (W - 1) - static_cast<int>(back);               // 0 .. W - 2
#pragma unroll
      for (int e = 0; e < 8; ++e)
        win[j][e] = ld1<BF16>(A.state, (static_cast<int64_t>(slot) * A.CD + c + e) * (W - 1) + idx);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) win[j][e] = 0.f;
    }
  }
}

// A block takes 256 consecutive channel groups of one 64-token run; its rows stream through
// a two-stage shared-memory ring filled by cp.async (each thread copies and later reads only
// its own 16-byte pieces, so no barrier is needed), keeping up to 128 KB of x in flight per SM.
template <bool BF16>
struct ConvRing {
  static constexpr int ROWS = BF16 ? 8 : 4;     // token rows per stage (64 KB: two CTAs per SM)
  static constexpr int PIECE = BF16 ? 16 : 32;  // bytes of 8 channels of one row
  static constexpr size_t bytes = 2 * ROWS * 256 * PIECE;
};

template <bool BF16, int W>
__global__ void __launch_bounds__(256, 2) conv_kernel(ConvArgs A) {
  using R = ConvRing<BF16>;
  extern __shared__ __align__(16) unsigned char ring[];
  const int tid = threadIdx.x;
  const int CG = A.CD / 8;
  const int ncb = (CG + 255) / 256;
  const int64_t runs = (A.T + kConvRun - 1) / kConvRun;
  const uint32_t ring_base = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  for (int64_t unit = blockIdx.x; unit < runs * ncb; unit += gridDim.x) {
    const int64_t r = unit / ncb;
    const int cgi = static_cast<int>(unit % ncb) * 256 + tid;
    const bool active = cgi < CG;
    const int c = active ? cgi * 8 : 0;
    const int64_t t_beg = r * kConvRun;
    const int64_t t_end = min(A.T, t_beg + kConvRun);
    const int nst = static_cast<int>((t_end - t_beg + R::ROWS - 1) / R::ROWS);
    auto piece = [&](int buf, int u) -> uint32_t {
      return ring_base + static_cast<uint32_t>(((buf * R::ROWS + u) * 256 + tid) * R::PIECE);
    };
    auto issue = [&](int st) {                  // stage st into buffer st % 2
#pragma unroll
      for (int u = 0; u < R::ROWS; ++u) {
        const int64_t t = t_beg + static_cast<int64_t>(st) * R::ROWS + u;
        if (active && t < t_end) {
          const unsigned char* src = static_cast<const unsigned char*>(A.x) +
                                     (t * A.CD + c) * (BF16 ? 2 : 4);
          tc_cp_async16(piece(st & 1, u), src);
          if constexpr (!BF16) tc_cp_async16(piece(st & 1, u) + 16, src + 16);
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    issue(0);
    if (nst > 1) issue(1);
    float wt[W][8], bs[8];
    int s = 0;
    int64_t bos = 0, eos = 0;
    float win[W > 1 ? W - 1 : 1][8];
    if (active) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
#pragma unroll
        for (int i = 0; i < W; ++i) wt[i][e] = A.w[static_cast<int64_t>(c + e) * W + i];
        bs[e] = A.bias ? A.bias[c + e] : 0.f;
      }
      s = seq_of(A.offsets, A.B, t_beg);
      bos = A.offsets ? A.offsets[s] : s;
      eos = A.offsets ? A.offsets[s + 1] : s + 1;
      fill_window<BF16, W>(A, s, bos, t_beg, c, win);
    }
    for (int st = 0; st < nst; ++st) {
      if (st + 1 < nst) asm volatile("cp.async.wait_group 1;" ::: "memory");
      else asm volatile("cp.async.wait_group 0;" ::: "memory");
      if (active) {
#pragma unroll 4
        for (int u = 0; u < R::ROWS; ++u) {
          const int64_t t = t_beg + static_cast<int64_t>(st) * R::ROWS + u;
          if (t >= t_end) break;
          if (t >= eos) {                       // the next (non-empty) sequence starts here
            s = seq_of(A.offsets, A.B, t);
            bos = A.offsets ? A.offsets[s] : s;
            eos = A.offsets ? A.offsets[s + 1] : s + 1;
            fill_window<BF16, W>(A, s, bos, t, c, win);
          }
          float cur[8], z[8];
          const unsigned char* sp = ring + ((st & 1) * R::ROWS + u) * 256 * R::PIECE + tid * R::PIECE;
          if constexpr (BF16) {
            const uint4 q = *reinterpret_cast<const uint4*>(sp);
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              cur[2 * e] = __uint_as_float(w4[e] << 16);
              cur[2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
            }
          } else {
            const float4 p0 = *reinterpret_cast<const float4*>(sp);
            const float4 p1 = *reinterpret_cast<const float4*>(sp + 16);
            cur[0] = p0.x; cur[1] = p0.y; cur[2] = p0.z; cur[3] = p0.w;
            cur[4] = p1.x; cur[5] = p1.y; cur[6] = p1.z; cur[7] = p1.w;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float acc = bs[e] + wt[W - 1][e] * cur[e];
#pragma unroll
            for (int j = 0; j < W - 1; ++j) acc += wt[j][e] * win[j][e];
            z[e] = silu<BF16>(acc);
          }
          st8<BF16>(A.y, t * A.CD + c, z);
#pragma unroll
          for (int j = 0; j + 1 < W - 1; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) win[j][e] = win[j + 1][e];
          if constexpr (W > 1)
#pragma unroll
            for (int e = 0; e < 8; ++e) win[W - 2][e] = cur[e];
        }
      }
      if (st + 2 < nst) issue(st + 2);          // this thread's pieces of the buffer are read
    }
  }
}

// the gates, elementwise: log-decay = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b);
// four consecutive elements per step (16-byte moves when every array is 16-byte aligned)
__device__ __forceinline__ float decay_gate(const ConvArgs& A, int64_t i) {
  const int hj = static_cast<int>(i % (A.HV * A.GW));
  const float zz = A.a[i] + (A.dt_bias ? A.dt_bias[hj] : 0.f);
  const float sp = zz > 20.f ? zz : log1pf(expf(zz));
  return A.A_log ? -expf(A.A_log[hj / A.GW]) * sp : -sp;
}

__global__ void __launch_bounds__(256) gates_kernel(ConvArgs A, bool vec) {
  const int64_t ng = A.T * A.HV * A.GW, nb = A.T * A.HV;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t q4 = (ng + 3) / 4, total = q4 + (nb + 3) / 4;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < total; it += stride) {
    if (it < q4) {
      const int64_t i0 = 4 * it;
      if (vec && i0 + 4 <= ng) {
        float4 out;
        out.x = decay_gate(A, i0);
        out.y = decay_gate(A, i0 + 1);
        out.z = decay_gate(A, i0 + 2);
        out.w = decay_gate(A, i0 + 3);
        *reinterpret_cast<float4*>(A.g + i0) = out;
      } else {
        for (int64_t i = i0; i < min(ng, i0 + 4); ++i) A.g[i] = decay_gate(A, i);
      }
    } else {
      const int64_t i0 = 4 * (it - q4);
      if (vec && i0 + 4 <= nb) {
        const float4 bb = *reinterpret_cast<const float4*>(A.b + i0);
        *reinterpret_cast<float4*>(A.beta + i0) =
            make_float4(1.f / (1.f + expf(-bb.x)), 1.f / (1.f + expf(-bb.y)),
                        1.f / (1.f + expf(-bb.z)), 1.f / (1.f + expf(-bb.w)));
      } else {
        for (int64_t i = i0; i < min(nb, i0 + 4); ++i) A.beta[i] = 1.f / (1.f + expf(-A.b[i]));
      }
    }
  }
}

// after the convolution: each touched slot takes its sequence's last W - 1 inputs (an empty
// sequence keeps its state; a sequence shorter than W - 1 shifts the old state in front)
template <bool BF16, int W>
__global__ void __launch_bounds__(256) conv_state_kernel(ConvArgs A) {
  const int CG = A.CD / 8;
  const int64_t items = static_cast<int64_t>(A.B) * CG;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < items;
       it += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int s = static_cast<int>(it / CG);
    const int c = static_cast<int>(it % CG) * 8;
    const int64_t bos = A.offsets ? A.offsets[s] : s;
    const int64_t eos = A.offsets ? A.offsets[s + 1] : s + 1;
    if (bos > eos || eos > A.T) {
      if (c == 0) raise_device_error(A.err, KDA_DEVERR_OFFSETS);
      continue;
    }
    const uint32_t slot = A.slot_idx[s];
    if (slot >= static_cast<uint32_t>(A.num_slots)) continue;   // reported by the conv kernel
    float ns[W - 1][8];
#pragma unroll
    for (int j = 0; j < W - 1; ++j) {
      const int64_t pos = eos - (W - 1) + j;
      if (pos >= bos) {
        ld8<BF16>(A.x, pos * A.CD + c, ns[j]);
      } else {
        const int idx = (W - 1) - static_cast<int>(bos - pos);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          ns[j][e] = ld1<BF16>(A.state, (static_cast<int64_t>(slot) * A.CD + c + e) * (W - 1) + idx);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
      for (int j = 0; j < W - 1; ++j) {
        const int64_t o = (static_cast<int64_t>(slot) * A.CD + c + e) * (W - 1) + j;
        if constexpr (BF16) static_cast<uint16_t*>(A.state)[o] = f32_to_bf16_bits(ns[j][e]);
        else static_cast<float*>(A.state)[o] = ns[j][e];
      }
  }
}

static unsigned conv_grid(int64_t items) {
  const int64_t blocks = (items + 255) / 256;
  return static_cast<unsigned>(blocks < 1 ? 1 : (blocks > 152 * 32 ? 152 * 32 : blocks));
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <bool BF16, int W>
static cudaError_t launch_conv_t(const ConvArgs& A, cudaStream_t st) {
  const int64_t runs = (A.T + kConvRun - 1) / kConvRun;
  const int64_t items = runs * (A.CD / 8);
  const int64_t gitems = (A.T * A.HV * A.GW + 3) / 4 + (A.T * A.HV + 3) / 4;
  cudaError_t e;
  if (gitems > 0) {
    const bool vec = aligned16(A.a) && aligned16(A.g) && aligned16(A.b) && aligned16(A.beta);
    gates_kernel<<<conv_grid(gitems), 256, 0, st>>>(A, vec);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (items > 0) {
    auto k = conv_kernel<BF16, W>;
    constexpr size_t smem = ConvRing<BF16>::bytes;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem))) != cudaSuccess)
      return e;
    const int64_t units = runs * ((A.CD / 8 + 255) / 256);
    k<<<static_cast<unsigned>(std::min<int64_t>(units, 152 * 8)), 256, smem, st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if constexpr (W > 1) {
    if (A.state && A.B > 0) {
      conv_state_kernel<BF16, W><<<conv_grid(static_cast<int64_t>(A.B) * (A.CD / 8)), 256, 0, st>>>(A);
      return cudaGetLastError();
    }
  }
  return cudaSuccess;
}

template <bool BF16>
static cudaError_t launch_conv_b(const ConvArgs& A, int W, cudaStream_t st) {
  switch (W) {
    case 1: return launch_conv_t<BF16, 1>(A, st);
    case 2: return launch_conv_t<BF16, 2>(A, st);
    case 3: return launch_conv_t<BF16, 3>(A, st);
    default: return launch_conv_t<BF16, 4>(A, st);
  }
}

cudaError_t launch_conv_gates(const void* x, const float* w, const float* bias, const float* a,
                              const float* b, const float* A_log, const float* dt_bias,
                              const uint32_t* offsets, const uint32_t* slot_idx, void* state,
                              void* y, float* g, float* beta, int64_t T, int B, int CD, int HV,
                              int GW, int num_slots, int W, bool bf16, int32_t* err,
                              cudaStream_t st) {
  const ConvArgs A{x, w, bias, a, b, A_log, dt_bias, offsets, slot_idx, state, y, g, beta,
                   T, B, CD, HV, GW, num_slots, err};
  return bf16 ? launch_conv_b<true>(A, W, st) : launch_conv_b<false>(A, W, st);
}

}  // namespace kda
