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
};

// The contractions over the value dimension of every (chunk, value head) on tensor cores
// (d = 128, chunk 64): dQ~, dK~, dK_end, dA, dM, dgamma and the first term of dbeta into the
// workspace, as bwd_vc_kernel computes them.  Returns cudaErrorNotSupported when an operand
// cannot be copied by TMA (d_o not 16-byte aligned), so the caller runs the CUDA-core kernel.
cudaError_t launch_bwd_vc_tc(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A,
                             cudaStream_t st);

// The scan on tensor cores (d = 128, chunk 64): a forward kernel recording each chunk's
// incoming state and corrected values, then a reverse kernel carrying the state gradient
// (dY, dV, the state gradients per chunk and w.r.t. the initial states), as bwd_scan_kernel
// computes them.  Needs the local stage's transposed copies (loc.KendT ... loc.TT); returns
// cudaErrorNotSupported when a tensor map cannot be encoded, so the caller runs the
// CUDA-core scan.
cudaError_t launch_bwd_scans_tc(const Problem& P, const BwdWorkspace& ws, const BwdArgs& A, bool sbf16,
                                cudaStream_t st);

}  // namespace kda
