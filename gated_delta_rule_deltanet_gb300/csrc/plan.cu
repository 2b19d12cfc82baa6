// plan.cu -- device-side validation of a ragged batch and its chunk table.
#include "prefill_plan.cuh"

namespace kda {

size_t plan_layout(const Problem& P, char* base, size_t off, PlanView* out) {
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? base + off : nullptr;
    off += (bytes + 255) & ~size_t(255);
    return p;
  };
  PlanView v;
  v.info = reinterpret_cast<int32_t*>(take(4 * sizeof(int32_t)));
  v.seq_chunk0 = reinterpret_cast<int32_t*>(take((static_cast<size_t>(P.num_seqs) + 1) * 4));
  v.chunks = reinterpret_cast<ChunkInfo*>(take(static_cast<size_t>(plan_max_chunks(P)) * sizeof(ChunkInfo)));
  v.seq_order = reinterpret_cast<int32_t*>(take(static_cast<size_t>(P.num_seqs) * sizeof(int32_t)));
  v.skip = reinterpret_cast<int32_t*>(take(static_cast<size_t>(P.num_seqs) * P.HV * sizeof(int32_t)));
  if (out) *out = v;
  return off;
}

constexpr int kPlanThreads = 1024;
static_assert(kPlanThreads == 32 * 32, "the plan's scan takes 32 warps of 32");

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(Problem P, PlanView plan, int max_chunks) {
  __shared__ int s_bad, s_longest;
  __shared__ int s_scan[kPlanThreads];
  __shared__ int s_n[kPlanThreads];            // chunks per sequence (B <= kPlanThreads)
  const int B = P.num_seqs, C = P.chunk, tid = threadIdx.x;
  if (tid == 0) {
    s_bad = 0;
    s_longest = 0;
  }
  for (int64_t u = tid; u < static_cast<int64_t>(B) * P.HV; u += kPlanThreads) plan.skip[u] = 0;
  __syncthreads();
  if (tid == 0 && (P.offsets[0] != 0u || static_cast<int64_t>(P.offsets[B]) != P.T)) atomicOr(&s_bad, 1);
  for (int b = tid; b < B; b += kPlanThreads) {
    if (P.offsets[b + 1] < P.offsets[b]) atomicOr(&s_bad, 1);
    if (P.slot_idx[b] >= static_cast<uint32_t>(P.num_slots)) atomicOr(&s_bad, 2);
  }
  if (P.flags & KDA_FLAG_CHECKED) {
    const int64_t pairs = static_cast<int64_t>(B) * B;
    for (int64_t pr = tid; pr < pairs; pr += kPlanThreads) {
      const int i = static_cast<int>(pr / B), j = static_cast<int>(pr % B);
      if (i < j && P.slot_idx[i] == P.slot_idx[j]) atomicOr(&s_bad, 4);
    }
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      raise_device_error(P.err, (s_bad & 1) ? KDA_DEVERR_OFFSETS
                                : (s_bad & 2) ? KDA_DEVERR_SLOT_RANGE : KDA_DEVERR_SLOT_DUP);
      plan.info[0] = 0;
      plan.info[1] = 0;
      plan.info[2] = 0;
    }
    return;
  }
  // chunk counts over a contiguous range of sequences per thread, then a block scan
  const int per = (B + kPlanThreads - 1) / kPlanThreads;
  const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
  int local = 0, longest = 0;
  for (int b = b0; b < b1; ++b) {
    const int nb = static_cast<int>((P.offsets[b + 1] - P.offsets[b] + C - 1) / C);
    local += nb;
    longest = max(longest, nb);
  }
  atomicMax(&s_longest, longest);
  // block-wide inclusive scan of `local`: within each warp by shuffles, then over the warp totals
  const int lane = tid & 31, warp = tid >> 5;
  int inc = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (lane == 31) s_scan[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = s_scan[lane];                       // kPlanThreads / 32 == 32 warp totals
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    s_scan[32 + lane] = w;                      // inclusive totals of warps 0..lane
  }
  __syncthreads();
  inc += warp > 0 ? s_scan[32 + warp - 1] : 0;
  if (tid == kPlanThreads - 1) s_scan[0] = inc;   // the grand total, read below
  __syncthreads();
  int base = inc - local;
  for (int b = b0; b < b1; ++b) {
    plan.seq_chunk0[b] = base;
    base += static_cast<int>((P.offsets[b + 1] - P.offsets[b] + C - 1) / C);
  }
  const int total = s_scan[0];
  if (tid == kPlanThreads - 1) plan.seq_chunk0[B] = total;
  __syncthreads();                              // the first chunk of every sequence is written
  // the sequences by decreasing chunk count: a sequence's rank is the number of sequences with
  // more chunks, or as many and a lower index
  if (B <= kPlanThreads) {
    if (tid < B) s_n[tid] = plan.seq_chunk0[tid + 1] - plan.seq_chunk0[tid];
    __syncthreads();
    if (tid < B) {
      const int nb = s_n[tid];
      int r = 0;
      for (int j = 0; j < B; ++j) r += (s_n[j] > nb) || (s_n[j] == nb && j < tid);
      plan.seq_order[r] = tid;
    }
  } else {
    for (int b = tid; b < B; b += kPlanThreads) plan.seq_order[b] = b;
  }
  // one table entry per thread and step: its sequence by binary search over the first chunks
  // (an empty sequence shares its first chunk with the next one)
  for (int g = tid; g < min(total, max_chunks); g += kPlanThreads) {
    int lo = 0, hi = B;                         // seq_chunk0[lo] <= g < seq_chunk0[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (plan.seq_chunk0[mid] <= g) lo = mid; else hi = mid;
    }
    const int c = g - plan.seq_chunk0[lo];
    const uint32_t bos = P.offsets[lo], len = P.offsets[lo + 1] - bos;
    ChunkInfo ci;
    ci.seq = lo;
    ci.n = static_cast<int32_t>(min(static_cast<uint32_t>(C), len - static_cast<uint32_t>(c * C)));
    ci.t0 = static_cast<int64_t>(bos) + static_cast<int64_t>(c) * C;
    plan.chunks[g] = ci;
  }
  if (tid == 0) {
    plan.info[0] = total;
    plan.info[1] = 1;
    plan.info[2] = s_longest;
  }
}

cudaError_t launch_plan(const Problem& P, const PlanView& plan, cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(P, plan, plan_max_chunks(P));
  return cudaGetLastError();
}

}  // namespace kda
