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
  float* Qt;    // [chunk][HV][C][D] (null in the backward's tensor-core path, which takes QtT)
  float* Kend;  // [chunk][HV][C][D]
  float* Aqk;   // [chunk][HV][C][C] (likewise, AqkT)
  float* gamma; // [chunk][HV][D]
  float* T;     // [chunk][HV][C][C] (I + A_kk)^-1, or null (kept only by the backward pass)
  float* Kt;    // [chunk][HV][C][D] K~ = k^ exp(G), or null (likewise)
  // transposed copies for the backward's tensor-core scans (K-major operands), or null:
  float* KendT; // [chunk][HV][D][C]
  float* QtT;   // [chunk][HV][D][C]
  float* WT;    // [chunk][HV][D][C]
  float* AqkT;  // [chunk][HV][C][C]
  float* TT;    // [chunk][HV][C][C]
  int32_t* local_fb;  // [chunk][HV] per-channel decay, tensor-core path: this chunk's decay left
                      // the anchored factors' range and the CUDA-core stage computes it
};

// 16-byte vector moves of N floats between registers and 16-byte aligned memory (scalar when
// N is not a multiple of 4)
template <int N>
__device__ __forceinline__ void ld_row(float (&x)[N], const float* p) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int e = 0; e < N; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + e);
      x[e] = v.x; x[e + 1] = v.y; x[e + 2] = v.z; x[e + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) x[e] = p[e];
  }
}

template <int N>
__device__ __forceinline__ void st_row(float* p, const float (&x)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int e = 0; e < N; e += 4)
      *reinterpret_cast<float4*>(p + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) p[e] = x[e];
  }
}

// 8 consecutive q/k/v elements (16-byte aligned: the rows are) widened to fp32
template <bool BF16>
__device__ __forceinline__ void load8(const void* base, int64_t i, float (&x)[8]) {
  if constexpr (BF16) {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  } else {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
    const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + i + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

template <int D, int C>
struct SimtLocalSmem {
  static constexpr int DP = D + 4;  // padded rows, 16-byte aligned
  static constexpr int CP = C + 4;
  static constexpr size_t floats = 4 * C * DP + 4 * C * CP + 3 * C + 2 * D;
  static constexpr size_t bytes = floats * sizeof(float);
};

// T = (I + A)^-1 for a strictly lower C x C matrix A (rows of CP floats in shared memory; s_T
// zero on entry): forward substitution inside each 16 x 16 diagonal block by one half-warp,
// then neighbouring blocks merged, T21 = -T22 (A21 T11), doubling the block size.  s_X is
// scratch.  Called by all NT threads; ends with a block barrier.
template <int C, int CP, int NT>
__device__ __forceinline__ void tri_unit_lower_inverse(const float* s_A, float* s_T, float* s_X, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
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
  for (int s = 16; s < C; s *= 2) {
    const int pairs = C / (2 * s);
    for (int idx = tid; idx < pairs * s * s; idx += NT) {
      const int p = idx / (s * s), r = (idx / s) % s, c = idx % s;
      const int rr = 2 * p * s + s, cc = 2 * p * s;
      float acc = 0.f;
      for (int m = c; m < s; ++m) acc += s_A[(rr + r) * CP + cc + m] * s_T[(cc + m) * CP + cc + c];
      s_X[(rr + r) * CP + cc + c] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < pairs * s * s; idx += NT) {
      const int p = idx / (s * s), r = (idx / s) % s, c = idx % s;
      const int rr = 2 * p * s + s, cc = 2 * p * s;
      float acc = 0.f;
      for (int m = 0; m <= r; ++m) acc += s_T[(rr + r) * CP + rr + m] * s_X[(rr + m) * CP + cc + c];
      s_T[(rr + r) * CP + cc + c] = -acc;
    }
    __syncthreads();
  }
}

// Per-channel decay spans at most this many nats between a token and the chunk's middle token
// for the anchored factors exp(G - G_a), exp(G_a - G) to be used (they stay far inside fp32);
// beyond it the pairwise decay is evaluated per pair and channel.
constexpr float kSimtAnchorRange = 80.f;

// Every thread owns tiles of rows r0 .. r0 + C/16 - 1 (r0 = (t / 16) C/16): of a C x C
// product the columns (t % 16) C/16 + b, of a C x D product the columns (t % 16) D/16 + b.
template <int D, int C, bool QBF16, bool PERCH>
// win: the chunks of one window of positions (the backward's bounded workspace), each in the
// workspace slot of its window; {0, 0} for every chunk in its own slot.
__global__ void __launch_bounds__(256) simt_local_kernel(Problem P, SimtWorkspace ws, ChunkWindow win,
                                                          int fb_only) {
  constexpr int NT = 256;
  constexpr int DP = SimtLocalSmem<D, C>::DP;
  constexpr int CP = SimtLocalSmem<D, C>::CP;
  constexpr int RT = C / 16, JA = C / 16, JC = D / 16;
  extern __shared__ __align__(16) float smem[];
  float* s_k = smem;              // [C][DP] normalised keys (K+ = k^ exp(G - G_a) once anchored)
  float* s_q = s_k + C * DP;      // [C][DP] normalised, scaled queries (Q+ likewise)
  float* s_v = s_q + C * DP;      // [C][DP] values
  float* s_G = s_v + C * DP;      // [C][DP] cumulative log-decay (column 0 when scalar);
                                  //   K- = k^ exp(G_a - G) once anchored
  float* s_A = s_G + C * DP;      // [C][CP] strictly lower beta K K^T (decayed)
  float* s_Aq = s_A + C * CP;     // [C][CP] lower Q K^T (decayed)
  float* s_T = s_Aq + C * CP;     // [C][CP] (I + A)^-1
  float* s_X = s_T + C * CP;      // [C][CP] merge temporaries
  float* s_beta = s_X + C * CP;   // [C]
  float* s_inv = s_beta + C;      // [2C] row scales of k and q
  float* s_ga = s_inv + 2 * C;    // [D] G_a, then exp(G_a)
  float* s_gl = s_ga + D;         // [D] G_last, then exp(G_last - G_a)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int gc;
  if (ws.plan.info[1] == 0 || !window_chunk(ws.plan, P.num_seqs, win, blockIdx.x, &gc)) return;
  // after the tensor-core local stage: only the chunks it left here
  if (fb_only && ws.local_fb[static_cast<int64_t>(blockIdx.x) * P.HV + blockIdx.y] == 0) return;
  const ChunkInfo ci = ws.plan.chunks[gc];
  const int h = blockIdx.y;
  const int HV = P.HV;
  const int kh = h / (HV / P.HK);
  const int n = ci.n;
  const int64_t t0 = ci.t0;
  // C x C products: thread columns (t % 16) + 16 b, so that the 8 threads of a quarter-warp read
  // 8 consecutive padded rows, whose 16-byte pieces fall on different banks
  const int r0 = (tid / 16) * RT, a0 = tid % 16, c0 = (tid % 16) * JC;
  // additive write (no delta rule): A_kk = 0 makes T = I, and W = 0
  const bool delta = !(P.flags & KDA_FLAG_NO_DELTA);

  for (int u = tid; u < C * (D / 8); u += NT) {
    const int i = u / (D / 8), c = (u % (D / 8)) * 8;
    float kx[8] = {}, qx[8] = {}, vx[8] = {}, gx[8] = {};
    if (i < n) {
      const int64_t t = t0 + i;
      load8<QBF16>(P.k, t * P.k_stride + static_cast<int64_t>(kh) * D + c, kx);
      load8<QBF16>(P.q, t * P.q_stride + static_cast<int64_t>(kh) * D + c, qx);
      load8<QBF16>(P.v, t * P.v_stride + static_cast<int64_t>(h) * D + c, vx);
      if (PERCH)
#pragma unroll
        for (int e = 0; e < 8; ++e) gx[e] = P.g[(t * HV + h) * D + c + e];
    }
    st_row(s_k + i * DP + c, kx);
    st_row(s_q + i * DP + c, qx);
    st_row(s_v + i * DP + c, vx);
    if (PERCH) st_row(s_G + i * DP + c, gx);
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
  } else if (warp == 0) {                       // warp scan, C / 32 rows per lane (one if C < 32)
    constexpr int RPL = C >= 32 ? C / 32 : 1;
    float loc[RPL];
    float tot = 0.f;
#pragma unroll
    for (int r = 0; r < RPL; ++r) {
      const int row = lane * RPL + r;
      loc[r] = row < C ? s_G[row * DP] : 0.f;
      tot += loc[r];
    }
    float inc = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    float acc = inc - tot;
#pragma unroll
    for (int r = 0; r < RPL; ++r) {
      const int row = lane * RPL + r;
      acc += loc[r];
      if (row < C) s_G[row * DP] = acc;
    }
  }
  __syncthreads();

  // per-channel decay: anchored factors at the middle token when the range allows
  bool anchored = false;
  if constexpr (PERCH) {
    const int am = (n - 1) / 2;
    for (int c = tid; c < D; c += NT) {
      s_ga[c] = s_G[am * DP + c];
      s_gl[c] = s_G[(C - 1) * DP + c];
    }
    __syncthreads();
    bool wide = false;
    for (int idx = tid; idx < C * D; idx += NT) {
      const int i = idx / D, c = idx % D;
      wide |= fabsf(s_G[i * DP + c] - s_ga[c]) > kSimtAnchorRange;
    }
    anchored = !__syncthreads_or(wide);
    if (anchored) {
      for (int idx = tid; idx < C * D; idx += NT) {
        const int i = idx / D, c = idx % D;
        const float d = s_G[i * DP + c] - s_ga[c];
        const float e = expf(d), r = expf(-d);
        s_q[i * DP + c] *= e;                   // Q+
        s_G[i * DP + c] = s_k[i * DP + c] * r;  // K-
        s_k[i * DP + c] *= e;                   // K+
      }
      __syncthreads();
    }
  }

  // A_kk (strictly lower, times beta_i) and A_qk (lower with diagonal)
  if (!PERCH || anchored) {
    const float* Km = PERCH ? s_G : s_k;
    float akk[RT][JA], aqk[RT][JA];
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int b = 0; b < JA; ++b) akk[a][b] = aqk[a][b] = 0.f;
#pragma unroll 2
    for (int c = 0; c < D; c += 4) {
      float4 ki[RT], qi[RT], kj[JA];
#pragma unroll
      for (int a = 0; a < RT; ++a) {
        ki[a] = *reinterpret_cast<const float4*>(s_k + (r0 + a) * DP + c);
        qi[a] = *reinterpret_cast<const float4*>(s_q + (r0 + a) * DP + c);
      }
#pragma unroll
      for (int b = 0; b < JA; ++b) kj[b] = *reinterpret_cast<const float4*>(Km + (a0 + 16 * b) * DP + c);
#pragma unroll
      for (int a = 0; a < RT; ++a)
#pragma unroll
        for (int b = 0; b < JA; ++b) {
          akk[a][b] += ki[a].x * kj[b].x + ki[a].y * kj[b].y + ki[a].z * kj[b].z + ki[a].w * kj[b].w;
          aqk[a][b] += qi[a].x * kj[b].x + qi[a].y * kj[b].y + qi[a].z * kj[b].z + qi[a].w * kj[b].w;
        }
    }
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int b = 0; b < JA; ++b) {
        const int i = r0 + a, j = a0 + 16 * b;
        const float dec = PERCH ? 1.f : (j <= i ? expf(s_G[i * DP] - s_G[j * DP]) : 0.f);
        s_A[i * CP + j] = (delta && j < i) ? s_beta[i] * (akk[a][b] * dec) : 0.f;
        s_Aq[i * CP + j] = j <= i ? aqk[a][b] * dec : 0.f;
      }
  } else {
    // exact per pair and channel: the cumulative decay exceeds the anchored range
    for (int idx = tid; idx < C * C; idx += NT) {
      const int i = idx / C, j = idx % C;
      float akk = 0.f, aqk = 0.f;
      if (j <= i) {
        for (int c = 0; c < D; ++c) {
          const float kj = s_k[j * DP + c] * expf(s_G[i * DP + c] - s_G[j * DP + c]);
          akk += s_k[i * DP + c] * kj;
          aqk += s_q[i * DP + c] * kj;
        }
      }
      s_A[i * CP + j] = (delta && j < i) ? s_beta[i] * akk : 0.f;
      s_Aq[i * CP + j] = aqk;
    }
  }
  __syncthreads();

  tri_unit_lower_inverse<C, CP, NT>(s_A, s_T, s_X, tid);

  const int64_t unit = static_cast<int64_t>(blockIdx.x) * HV + h;
  float* gW = ws.W + unit * C * D;
  float* gU = ws.U + unit * C * D;
  float* gQ = ws.Qt ? ws.Qt + unit * C * D : nullptr;
  float* gK = ws.Kend + unit * C * D;
  if (PERCH && anchored) {
    for (int c = tid; c < D; c += NT) {
      const float ga = s_ga[c], gl = s_gl[c];
      ws.gamma[unit * D + c] = expf(gl);
      s_ga[c] = expf(ga);                       // K~ = K+ exp(G_a), Q~ = Q+ exp(G_a)
      s_gl[c] = expf(gl - ga);                  // K_end = K- exp(G_last - G_a)
    }
    __syncthreads();
  } else {
    for (int c = tid; c < D; c += NT)
      ws.gamma[unit * D + c] = expf(PERCH ? s_G[(C - 1) * DP + c] : s_G[(C - 1) * DP]);
  }
  // boundary-decayed queries, keys decayed to the chunk end, and the right-hand sides
  // beta k exp(G) (into s_q) and beta v (in place), each thread its own tile
#pragma unroll
  for (int a = 0; a < RT; ++a) {
    const int i = r0 + a;
    const float bi = s_beta[i];
    float qt[JC], ke[JC], kt[JC];
#pragma unroll
    for (int b = 0; b < JC; ++b) {
      const int c = c0 + b;
      if (PERCH && anchored) {
        qt[b] = s_q[i * DP + c] * s_ga[c];
        kt[b] = s_k[i * DP + c] * s_ga[c];
        ke[b] = s_G[i * DP + c] * s_gl[c];
      } else {
        const float Gi = PERCH ? s_G[i * DP + c] : s_G[i * DP];
        const float Gl = PERCH ? s_G[(C - 1) * DP + c] : s_G[(C - 1) * DP];
        const float di = expf(Gi);
        qt[b] = s_q[i * DP + c] * di;
        kt[b] = s_k[i * DP + c] * di;
        ke[b] = s_k[i * DP + c] * expf(Gl - Gi);
      }
    }
    if (gQ) st_row(gQ + i * D + c0, qt);
    if (ws.Kt) st_row(ws.Kt + unit * C * D + i * D + c0, kt);
    if (ws.KendT) {                             // the backward's tf32 operands, rounded to nearest
#pragma unroll
      for (int b = 0; b < JC; ++b) {
        ke[b] = tf32_nearest(ke[b]);
        ws.KendT[(unit * D + c0 + b) * C + i] = ke[b];
        ws.QtT[(unit * D + c0 + b) * C + i] = tf32_nearest(qt[b]);
      }
    }
    st_row(gK + i * D + c0, ke);
#pragma unroll
    for (int b = 0; b < JC; ++b) {
      s_q[i * DP + c0 + b] = delta ? bi * kt[b] : 0.f;
      s_v[i * DP + c0 + b] *= bi;
    }
  }
  if (ws.Aqk)
    for (int idx = tid; idx < C * C; idx += NT) ws.Aqk[unit * C * C + idx] = s_Aq[(idx / C) * CP + idx % C];
  if (ws.T)
    for (int idx = tid; idx < C * C; idx += NT) ws.T[unit * C * C + idx] = s_T[(idx / C) * CP + idx % C];
  if (ws.TT)
    for (int idx = tid; idx < C * C; idx += NT) {
      ws.TT[unit * C * C + idx] = tf32_nearest(s_T[(idx % C) * CP + idx / C]);
      ws.AqkT[unit * C * C + idx] = tf32_nearest(s_Aq[(idx % C) * CP + idx / C]);
    }
  __syncthreads();
  // W = T (beta k exp(G)),  U = T (beta v)
  float w[RT][JC], uu[RT][JC];
#pragma unroll
  for (int a = 0; a < RT; ++a)
#pragma unroll
    for (int b = 0; b < JC; ++b) w[a][b] = uu[a][b] = 0.f;
  for (int j = 0; j < r0 + RT; ++j) {           // T is lower triangular: rows r0.. need j < r0 + RT
    float tq[JC], tv[JC];
    ld_row(tq, s_q + j * DP + c0);
    ld_row(tv, s_v + j * DP + c0);
#pragma unroll
    for (int a = 0; a < RT; ++a) {
      const float t = s_T[(r0 + a) * CP + j];
#pragma unroll
      for (int b = 0; b < JC; ++b) {
        w[a][b] += t * tq[b];
        uu[a][b] += t * tv[b];
      }
    }
  }
  if (ws.WT) {                                  // the backward's tf32 operands, rounded to nearest
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int b = 0; b < JC; ++b) w[a][b] = tf32_nearest(w[a][b]);
#pragma unroll
    for (int b = 0; b < JC; ++b) {
      float col[RT];
#pragma unroll
      for (int a = 0; a < RT; ++a) col[a] = w[a][b];
      st_row(ws.WT + (unit * D + c0 + b) * C + r0, col);
    }
  }
#pragma unroll
  for (int a = 0; a < RT; ++a) {
    st_row(gW + (r0 + a) * D + c0, w[a]);
    st_row(gU + (r0 + a) * D + c0, uu[a]);
  }
}

}  // namespace kda
