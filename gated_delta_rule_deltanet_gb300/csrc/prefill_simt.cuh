// prefill_simt.cuh -- the chunk-local stage of the CUDA-core prefill, shared with the
// backward pass (which reruns it and keeps two more of its results).
#pragma once

#include "kda_common.cuh"
#include "prefill_plan.cuh"

namespace kda {

struct SimtWorkspace {
  PlanView plan;
  float* W;     // [chunk][HV][C][D]
  float* U;     // [chunk][HV][C][D]
  float* Qt;    // [chunk][HV][C][D]
  float* Kend;  // [chunk][HV][C][D]
  float* Aqk;   // [chunk][HV][C][C]
  float* gamma; // [chunk][HV][D]
  float* T;     // [chunk][HV][C][C] (I + A_kk)^-1, or null (kept only by the backward pass)
  float* Kt;    // [chunk][HV][C][D] K~ = k^ exp(G), or null (likewise)
};

template <int D, int C>
struct SimtLocalSmem {
  static constexpr int DP = D + 1;  // padded rows: pair loops read column c of many rows
  static constexpr int CP = C + 1;
  static constexpr size_t floats = 4 * C * DP + 4 * C * CP + 3 * C;
  static constexpr size_t bytes = floats * sizeof(float);
};

template <int D, int C, bool QBF16, bool PERCH>
__global__ void __launch_bounds__(256) simt_local_kernel(Problem P, SimtWorkspace ws) {
  constexpr int NT = 256;
  constexpr int DP = SimtLocalSmem<D, C>::DP;
  constexpr int CP = SimtLocalSmem<D, C>::CP;
  extern __shared__ float smem[];
  float* s_k = smem;              // [C][DP] normalised keys
  float* s_q = s_k + C * DP;      // [C][DP] normalised, scaled queries
  float* s_v = s_q + C * DP;      // [C][DP] values
  float* s_G = s_v + C * DP;      // [C][DP] cumulative log-decay (column 0 when scalar)
  float* s_A = s_G + C * DP;      // [C][CP] strictly lower beta K K^T (decayed)
  float* s_Aq = s_A + C * CP;     // [C][CP] lower Q K^T (decayed)
  float* s_T = s_Aq + C * CP;     // [C][CP] (I + A)^-1
  float* s_X = s_T + C * CP;      // [C][CP] merge temporaries
  float* s_beta = s_X + C * CP;   // [C]
  float* s_inv = s_beta + C;      // [2C] row scales of k and q

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (ws.plan.info[1] == 0 || static_cast<int>(blockIdx.x) >= ws.plan.info[0]) return;
  const ChunkInfo ci = ws.plan.chunks[blockIdx.x];
  const int h = blockIdx.y;
  const int HV = P.HV;
  const int kh = h / (HV / P.HK);
  const int n = ci.n;
  const int64_t t0 = ci.t0;
  // additive write (no delta rule): A_kk = 0 makes T = I, and W = 0
  const bool delta = !(P.flags & KDA_FLAG_NO_DELTA);

  for (int idx = tid; idx < C * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    float kv = 0.f, qv = 0.f, vv = 0.f, gv = 0.f;
    if (i < n) {
      const int64_t t = t0 + i;
      kv = load_elem<QBF16>(P.k, t * P.k_stride + static_cast<int64_t>(kh) * D + c);
      qv = load_elem<QBF16>(P.q, t * P.q_stride + static_cast<int64_t>(kh) * D + c);
      vv = load_elem<QBF16>(P.v, t * P.v_stride + static_cast<int64_t>(h) * D + c);
      if (PERCH) gv = P.g[(t * HV + h) * D + c];
    }
    s_k[i * DP + c] = kv;
    s_q[i * DP + c] = qv;
    s_v[i * DP + c] = vv;
    if (PERCH) s_G[i * DP + c] = gv;
  }
  for (int i = tid; i < C; i += NT) {
    const bool live = i < n;
    s_beta[i] = live ? P.beta[(t0 + i) * HV + h] : 0.f;
    if (!PERCH) s_G[i * DP] = live ? P.g[(t0 + i) * HV + h] : 0.f;
  }
  for (int idx = tid; idx < C * CP; idx += NT) s_T[idx] = 0.f;
  __syncthreads();

  // L2 norms (one warp per row) and the query scale
  for (int i = warp; i < C; i += NT / 32) {
    float sk = 0.f, sq = 0.f;
    for (int c = lane; c < D; c += 32) {
      sk += s_k[i * DP + c] * s_k[i * DP + c];
      sq += s_q[i * DP + c] * s_q[i * DP + c];
    }
    sk = warp_sum(sk);
    sq = warp_sum(sq);
    if (lane == 0) {
      s_inv[i] = P.l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
      s_inv[C + i] = (P.l2norm ? rsqrtf(sq + 1e-6f) : 1.f) * P.scale;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < C * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    s_k[i * DP + c] *= s_inv[i];
    s_q[i * DP + c] *= s_inv[C + i];
  }
  // in-chunk inclusive cumulative log-decay; padded rows add nothing
  if (PERCH) {
    for (int c = tid; c < D; c += NT) {
      float acc = 0.f;
      for (int i = 0; i < C; ++i) {
        acc += s_G[i * DP + c];
        s_G[i * DP + c] = acc;
      }
    }
  } else if (tid == 0) {
    float acc = 0.f;
    for (int i = 0; i < C; ++i) {
      acc += s_G[i * DP];
      s_G[i * DP] = acc;
    }
  }
  __syncthreads();

  // A_kk (strictly lower, times beta_i) and A_qk (lower with diagonal)
  for (int idx = tid; idx < C * C; idx += NT) {
    const int i = idx / C, j = idx % C;
    float akk = 0.f, aqk = 0.f;
    if (j <= i) {
      if (PERCH) {
        for (int c = 0; c < D; ++c) {
          const float kj = s_k[j * DP + c] * expf(s_G[i * DP + c] - s_G[j * DP + c]);
          akk += s_k[i * DP + c] * kj;
          aqk += s_q[i * DP + c] * kj;
        }
      } else {
        for (int c = 0; c < D; ++c) {
          akk += s_k[i * DP + c] * s_k[j * DP + c];
          aqk += s_q[i * DP + c] * s_k[j * DP + c];
        }
        const float dec = expf(s_G[i * DP] - s_G[j * DP]);
        akk *= dec;
        aqk *= dec;
      }
    }
    s_A[i * CP + j] = (delta && j < i) ? s_beta[i] * akk : 0.f;
    s_Aq[i * CP + j] = aqk;
  }
  __syncthreads();

  // T = (I + A)^-1: forward substitution inside each 16x16 diagonal block ...
  if (warp < C / 16 && lane < 16) {
    const int base = warp * 16, col = base + lane;
    for (int r = 0; r < 16; ++r) {
      const int row = base + r;
      float val = r == lane ? 1.f : 0.f;
      for (int m = lane; m < r; ++m) val -= s_A[row * CP + base + m] * s_T[(base + m) * CP + col];
      s_T[row * CP + col] = r >= lane ? val : 0.f;
      __syncwarp(0x0000ffffu);
    }
  }
  __syncthreads();
  // ... then merge neighbours: T21 = -T22 (A21 T11), doubling the block size
  for (int s = 16; s < C; s *= 2) {
    const int pairs = C / (2 * s);
    for (int idx = tid; idx < pairs * s * s; idx += NT) {
      const int p = idx / (s * s), r = (idx / s) % s, c = idx % s;
      const int r0 = 2 * p * s + s, c0 = 2 * p * s;
      float acc = 0.f;
      for (int m = c; m < s; ++m) acc += s_A[(r0 + r) * CP + c0 + m] * s_T[(c0 + m) * CP + c0 + c];
      s_X[(r0 + r) * CP + c0 + c] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < pairs * s * s; idx += NT) {
      const int p = idx / (s * s), r = (idx / s) % s, c = idx % s;
      const int r0 = 2 * p * s + s, c0 = 2 * p * s;
      float acc = 0.f;
      for (int m = 0; m <= r; ++m) acc += s_T[(r0 + r) * CP + r0 + m] * s_X[(r0 + m) * CP + c0 + c];
      s_T[(r0 + r) * CP + c0 + c] = -acc;
    }
    __syncthreads();
  }

  const int64_t unit = static_cast<int64_t>(blockIdx.x) * HV + h;
  float* gW = ws.W + unit * C * D;
  float* gU = ws.U + unit * C * D;
  float* gQ = ws.Qt + unit * C * D;
  float* gK = ws.Kend + unit * C * D;
  // boundary-decayed queries, keys decayed to the chunk end, and the
  // right-hand sides beta k exp(G) (into s_q) and beta v (in place)
  for (int idx = tid; idx < C * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    const float Gi = PERCH ? s_G[i * DP + c] : s_G[i * DP];
    const float Gl = PERCH ? s_G[(C - 1) * DP + c] : s_G[(C - 1) * DP];
    const float di = expf(Gi);
    gQ[idx] = s_q[i * DP + c] * di;
    gK[idx] = s_k[i * DP + c] * expf(Gl - Gi);
    if (ws.Kt) ws.Kt[unit * C * D + idx] = s_k[i * DP + c] * di;
    s_q[i * DP + c] = delta ? s_beta[i] * s_k[i * DP + c] * di : 0.f;
    s_v[i * DP + c] *= s_beta[i];
  }
  for (int c = tid; c < D; c += NT)
    ws.gamma[unit * D + c] = expf(PERCH ? s_G[(C - 1) * DP + c] : s_G[(C - 1) * DP]);
  for (int idx = tid; idx < C * C; idx += NT) ws.Aqk[unit * C * C + idx] = s_Aq[(idx / C) * CP + idx % C];
  if (ws.T)
    for (int idx = tid; idx < C * C; idx += NT) ws.T[unit * C * C + idx] = s_T[(idx / C) * CP + idx % C];
  __syncthreads();
  // W = T (beta k exp(G)),  U = T (beta v)
  for (int idx = tid; idx < C * D; idx += NT) {
    const int i = idx / D, c = idx % D;
    float w = 0.f, u = 0.f;
    for (int j = 0; j <= i; ++j) {
      const float t = s_T[i * CP + j];
      w += t * s_q[j * DP + c];
      u += t * s_v[j * DP + c];
    }
    gW[idx] = w;
    gU[idx] = u;
  }
}

}  // namespace kda
