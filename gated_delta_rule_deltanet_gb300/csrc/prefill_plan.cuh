// prefill_plan.cuh -- the ragged chunk table shared by the prefill paths.
//
// Chunks restart at every sequence start, so a sequence of length L owns
// ceil(L / C) chunks and only its last one may be partial.  The table is
// built on the device from input_row_offsets (the host never sees the
// offsets, so no synchronisation is needed); its size is bounded on the host
// by T / C + B, which sizes the grids of the chunk-parallel kernels.
#pragma once

#include "kda_common.cuh"

namespace kda {

struct ChunkInfo {
  int32_t seq;  // sequence index b
  int32_t n;    // tokens in this chunk (1..C)
  int64_t t0;   // first token (row of the token-major tensors)
};

struct PlanView {
  int32_t* info;        // [0] chunks in the table, [1] 1 if the batch is valid, [2] chunks of
                        // the longest sequence
  int32_t* seq_chunk0;  // [B + 1] first chunk of each sequence (prefix sums)
  ChunkInfo* chunks;    // [max_chunks]
  int32_t* seq_order;   // [B] the sequences by decreasing chunk count (ties by index) when B is
                        // at most 1024, else in index order: the chain kernel starts its CTAs in
                        // this order, so that the longest scans are not left to a last wave
  int32_t* skip;        // [B * HV] nonzero: a kernel found this (sequence, value head) outside
                        // the tensor-core path's domain; the kernels that write o and the
                        // state pool leave it untouched (zeroed by the plan kernel)
};

// A window of chunk positions: every sequence's chunks w * wc .. w * wc + wc - 1 (counted from
// its start), chunk j of sequence b in slot b * wc + (j - w * wc).  wc == 0: every chunk of the
// table, in the slot of its own index.
struct ChunkWindow {
  int32_t w, wc;
};

// The chunk in `slot` of window `win`, or false when the slot holds none.
__device__ __forceinline__ bool window_chunk(const PlanView& plan, int num_seqs, ChunkWindow win, int slot,
                                            int* chunk) {
  if (win.wc == 0) {
    *chunk = slot;
    return slot < plan.info[0];
  }
  const int b = slot / win.wc, j = win.w * win.wc + slot % win.wc;
  if (b >= num_seqs) return false;
  const int c = plan.seq_chunk0[b] + j;
  *chunk = c;
  return c < plan.seq_chunk0[b + 1];
}

inline int plan_max_chunks(const Problem& P) {
  return static_cast<int>(P.T / P.chunk) + P.num_seqs;
}

// Carves the plan's arrays from `base` starting at byte `off` (256-aligned
// pieces); returns the new offset.  base == nullptr only measures.
size_t plan_layout(const Problem& P, char* base, size_t off, PlanView* out);

// Validates offsets / slots and builds the chunk table (one CTA).
cudaError_t launch_plan(const Problem& P, const PlanView& plan, cudaStream_t stream);

}  // namespace kda
