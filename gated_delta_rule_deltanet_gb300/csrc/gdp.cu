// gdp.cu -- Gated DeltaProduct as the gated delta rule over a virtual sequence.
//
// "Linear attention visualized", Gated Delta Product section: every token carries n_h
// transitions (its own key, value and gate each), the previous state decays once before
// the first, and the query reads after the last.  The page's virtual-sequence table maps
// substep j of token t to position m = t n_h + j of an ordinary gated-delta-rule sequence
// with key k_{t,j}, value v_{t,j}, gate beta_{t,j}, decay a_t at j = 0 and 1 after, query
// q_t at j = n_h - 1 and 0 before, and keeps every n_h-th output.
//
// With k, v and beta laid out [T, n_h, ...] they already are the virtual sequence's
// token-major tensors; only the query, the log-decay and the offsets need the expansion
// below, and the output the gather.  Everything in between is the library's own prefill.
#include "kda_common.cuh"

namespace kda {

// One thread per 16-byte piece of the virtual query rows, then one per element of the
// virtual log-decay rows, then one per offset.  qrow = HK * D elements, grow = HV (scalar)
// or HV * D.  offsets == nullptr means one token per sequence (the decode form).
template <bool QBF16>
__global__ void gdp_expand_kernel(const void* __restrict__ q, int64_t q_stride, const float* __restrict__ g,
                                  const uint32_t* __restrict__ offsets, int64_t T, int n_h,
                                  int64_t qrow, int64_t grow, int num_seqs, void* __restrict__ qv,
                                  float* __restrict__ gv, uint32_t* __restrict__ offv) {
  constexpr int QE = QBF16 ? 8 : 4;             // elements per 16-byte piece
  const int64_t qpieces = T * n_h * (qrow / QE);
  const int64_t gpieces = T * n_h * grow;
  const int64_t total = qpieces + gpieces + num_seqs + 1;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (i < qpieces) {
      const int64_t m = i / (qrow / QE), e = (i % (qrow / QE)) * QE;   // virtual row, element
      const int64_t t = m / n_h;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (m % n_h == n_h - 1) {
        const unsigned char* src = static_cast<const unsigned char*>(q) +
                                   (t * q_stride + e) * (QBF16 ? 2 : 4);
        val = *reinterpret_cast<const uint4*>(src);
      }
      *reinterpret_cast<uint4*>(static_cast<unsigned char*>(qv) + (m * qrow + e) * (QBF16 ? 2 : 4)) = val;
    } else if (i < qpieces + gpieces) {
      const int64_t r = i - qpieces;              // one element (a scalar gate row may be short)
      const int64_t m = r / grow, e = r % grow;
      gv[m * grow + e] = (m % n_h == 0) ? g[(m / n_h) * grow + e] : 0.f;
    } else {
      const int64_t b = i - qpieces - gpieces;   // 0..num_seqs
      offv[b] = offsets ? offsets[b] * static_cast<uint32_t>(n_h) : static_cast<uint32_t>(b * n_h);
    }
  }
}

// o[t] = ov[t n_h + n_h - 1], one thread per 16-byte piece (orow = HV * D fp32).
__global__ void gdp_gather_kernel(const float* __restrict__ ov, int64_t T, int n_h, int64_t orow,
                                  float* __restrict__ o) {
  const int64_t pieces = T * (orow / 4);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < pieces;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / (orow / 4), e = (i % (orow / 4)) * 4;
    *reinterpret_cast<float4*>(o + t * orow + e) =
        *reinterpret_cast<const float4*>(ov + (t * n_h + n_h - 1) * orow + e);
  }
}

static unsigned grid_for(int64_t work) {
  const int64_t blocks = (work + 255) / 256;
  return static_cast<unsigned>(blocks < 1 ? 1 : (blocks > 152 * 16 ? 152 * 16 : blocks));
}

cudaError_t launch_gdp_expand(const void* q, int64_t q_stride, bool qbf16, const float* g,
                              const uint32_t* offsets, int64_t T, int n_h, int64_t qrow,
                              int64_t grow, int num_seqs, void* qv, float* gv, uint32_t* offv,
                              cudaStream_t st) {
  const int64_t work = T * n_h * (qrow / (qbf16 ? 8 : 4) + grow) + num_seqs + 1;
  if (qbf16)
    gdp_expand_kernel<true><<<grid_for(work), 256, 0, st>>>(q, q_stride, g, offsets, T, n_h, qrow, grow,
                                                            num_seqs, qv, gv, offv);
  else
    gdp_expand_kernel<false><<<grid_for(work), 256, 0, st>>>(q, q_stride, g, offsets, T, n_h, qrow, grow,
                                                             num_seqs, qv, gv, offv);
  return cudaGetLastError();
}

cudaError_t launch_gdp_gather(const float* ov, int64_t T, int n_h, int64_t orow, float* o,
                              cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  gdp_gather_kernel<<<grid_for(T * (orow / 4)), 256, 0, st>>>(ov, T, n_h, orow, o);
  return cudaGetLastError();
}

}  // namespace kda
