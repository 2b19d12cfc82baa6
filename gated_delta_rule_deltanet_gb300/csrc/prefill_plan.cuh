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
                        // at most 1024, else in index order: the per-sequence scans start their
                        // CTAs in this order, so that the longest scans are not left to a last wave
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

// The per-sequence scans (one CTA per sequence, value head and value tile) run on a 1-D grid of
// B x HV x NVT CTAs, taken in the plan's order of decreasing sequence length: CTAs start in
// linear order, so the longest scans start first and the short ones fill in behind them.
struct SeqHeadTile {
  int b, h, vt;
};
__device__ __forceinline__ SeqHeadTile seq_head_tile(const PlanView& plan, int HV, int NVT) {
  const int L = static_cast<int>(blockIdx.x);
  return {plan.seq_order[L / (NVT * HV)], (L / NVT) % HV, L % NVT};
}
// The grid of seq_head_tile, or 0 CTAs when it would not fit a 1-D grid.
inline unsigned seq_head_tile_ctas(const Problem& P, int NVT) {
  const int64_t n = static_cast<int64_t>(P.num_seqs) * P.HV * NVT;
  return n > 0x7fffffff ? 0u : static_cast<unsigned>(n);
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
