// backward.cuh -- the backward pass's workspace and arguments, shared by its CUDA-core
// kernels (backward.cu) and its tensor-core kernels (backward_tc.cu).
#pragma once

#include "prefill_simt.cuh"

namespace kda {

struct BwdArgs {
  const float* d_o;      // [T, HV, D]
  const float* d_state;  // [num_slots, HV, D, D] or null: gradient w.r.t. the final states
  float* dq;             // [T, HK, D]
  float* dk;             // [T, HK, D]
  float* dv;             // [T, HV, D]
  float* dbeta;          // [T, HV]
  float* dg;             // [T, HV] or [T, HV, D]
  float* d_state0;       // [num_slots, HV, D, D] or null: gradient w.r.t. the initial states
};

struct BwdWorkspace {
  SimtWorkspace loc;
  float* Sck;   // [chunk][HV][D][D] state entering the chunk
  float* dSck;  // [chunk][HV][D][D] gradient w.r.t. the state leaving the chunk
  float* E;     // [chunk][HV][C][D] corrected values
  float* dY;    // [chunk][HV][C][D] T^T dE (rows past the chunk's end zero)
  float* dQt;   // [chunk][HV][C][D]
  float* dKt;   // [chunk][HV][C][D]
  float* dKe;   // [chunk][HV][C][D]
  float* dA;    // [chunk][HV][C][C]
  float* dM;    // [chunk][HV][C][C]
  float* dgam;  // [chunk][HV][D]
  float* dbr;   // [chunk][HV][C]
  // bounded workspace (windows of chunk positions; "chunk" above is then a window slot):
  int32_t* pair_fb;  // [chunk][HK] tensor-core path, per-channel decay: the pairwise terms of
                     // this (chunk, key head) are left to the CUDA-core kernel
  float* ckpt;  // [entry][HV][D][D] the state entering each window after a sequence's first
  float* carry; // [num_seqs][HV][D][D] the state gradient handed from window to window
};

// The contractions over the value dimension of every (chunk, value head) on tensor cores
// (d = 128, chunk 64): dQ~, dK~, dK_end, dA, dM, dgamma and the first term of dbeta into the
// workspace, as bwd_vc_kernel computes them.  Returns cudaErrorNotSupported when an operand
// cannot be copied by TMA (d_o not 16-byte aligned), so the caller runs the CUDA-core kernel.
cudaError_t launch_bwd_vc_tc(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A, ChunkWindow win,
                             int slots, cudaStream_t st);

// The scan on tensor cores (d = 128, chunk 64): a forward kernel recording each chunk's
// incoming state and corrected values, then a reverse kernel carrying the state gradient
// (dY, dV, the state gradients per chunk and w.r.t. the initial states), as bwd_scan_kernel
// computes them.  Needs the local stage's transposed copies (loc.KendT ... loc.TT); returns
// cudaErrorNotSupported when a tensor map cannot be encoded, so the caller runs the
// CUDA-core scan.
//
// Windowed (win.wc > 0, `slots` window slots): the chunks of window win.w only.  With
// record = false the forward kernel only carries the state through the window and stores it
// as the next window's checkpoint, and the reverse kernel does not run (the checkpoint sweep);
// with record = true both run as above, the state entering the window from its checkpoint
// and the state gradient handed on through ws.carry.
cudaError_t launch_bwd_scans_tc(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A, bool sbf16,
                                ChunkWindow win, int slots, bool record, cudaStream_t st);

// The chunk-local stage on tensor cores (d = 128, chunk 64, bf16 q/k/v): the workspace arrays
// simt_local_kernel writes for the tensor-core scans.  Per-channel decay (perch): with factors
// anchored at each chunk's middle token; a chunk whose decay leaves the anchor's range is
// flagged in ws.local_fb and left to simt_local_kernel.
cudaError_t launch_bwd_local_tc(const Problem& P, const SimtWorkspace& ws, ChunkWindow win, int slots,
                                bool perch, cudaStream_t st);

// The pairwise terms, dg, dbeta, dq and dk on tensor cores (d = 128, chunk 64, bf16 q/k), as
// bwd_pair_kernel computes them.  Per-channel decay (perch): with factors anchored at each
// chunk's middle token; a (chunk, key head) whose decay leaves the anchor's range is flagged in
// ws.pair_fb and left to bwd_pair_kernel.
cudaError_t launch_bwd_pair_tc(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A, ChunkWindow win,
                               int slots, bool perch, cudaStream_t st);

// index of the checkpoint of window w >= 1 of the sequence whose first chunk is c0
__host__ __device__ __forceinline__ int64_t ckpt_entry(int c0, ChunkWindow win) {
  return static_cast<int64_t>(c0 / win.wc) + win.w - 1;
}

}  // namespace kda
