// api.cu -- the C ABI: argument validation, workspace sizing and dispatch.
//
// Validation follows the argument checks of the chunked DeltaNet launcher in
// "From Attention to Learned Memory" (sec. 4: shapes, dtypes, chunk size in
// {16, 32, 64}), extended to the ragged batch, GQA ratio and slot pool of the
// Modular "gated_delta" module.  Everything here runs on the host before any
// launch; device-only checks live in the plan and decode kernels.
#include <mutex>

#include "kda_common.cuh"

namespace kda {
cudaError_t launch_decode(const Problem& P, bool qbf16, bool sbf16, bool perch, cudaStream_t s,
                          const Stages& st);
cudaError_t launch_prefill_simt(const Problem& P, void* workspace, bool qbf16, bool perch,
                                bool sbf16, cudaStream_t stream, const Stages& st);
size_t simt_workspace_bytes(const Problem& P);
bool tc_prefill_supported(const Problem& P, bool qbf16);
size_t tc_workspace_bytes(const Problem& P);
cudaError_t launch_prefill_tc(const Problem& P, void* workspace, bool perch, bool sbf16,
                              cudaStream_t stream, const Stages& st);
size_t split_workspace_bytes(const Problem& P);
cudaError_t launch_prefill_split(const Problem& P, void* workspace, bool perch, bool sbf16,
                                 cudaStream_t stream, const Stages& st);
int ring_record_elems(int D, bool perch);
cudaError_t launch_verify(const Problem& P, int window, float* ring, bool qbf16, bool sbf16,
                          bool perch, cudaStream_t stream);
cudaError_t launch_fold(const Problem& P, int window, const float* ring, const uint32_t* accepted,
                        bool sbf16, bool perch, cudaStream_t stream);
cudaError_t launch_gdp_expand(const void* q, int64_t q_stride, bool qbf16, const float* g,
                              const uint32_t* offsets, int64_t T, int n_h, int64_t qrow,
                              int64_t grow, int num_seqs, void* qv, float* gv, uint32_t* offv,
                              cudaStream_t st);
cudaError_t launch_gdp_gather(const float* ov, int64_t T, int n_h, int64_t orow, float* o,
                              cudaStream_t st);
cudaError_t launch_conv_gates(const void* x, const float* w, const float* bias, const float* a,
                              const float* b, const float* A_log, const float* dt_bias,
                              const uint32_t* offsets, const uint32_t* slot_idx, void* state,
                              void* y, float* g, float* beta, int64_t T, int B, int CD, int HV,
                              int GW, int num_slots, int W, bool bf16, int32_t* err,
                              cudaStream_t st);
size_t bwd_workspace_bytes(const Problem& P, bool qbf16, bool compact);
cudaError_t launch_prefill_bwd(const Problem& P, void* workspace, const float* d_o,
                               const float* d_state, float* dq, float* dk, float* dv,
                               float* dbeta, float* dg, float* d_state0, bool qbf16, bool perch,
                               bool sbf16, bool compact, cudaStream_t stream);
}  // namespace kda

using kda::Problem;

static_assert(sizeof(kda_params_t) == 88, "kda_params_t layout is part of the ABI");

// The device error word (one per device that loads the library).
__device__ int32_t g_kda_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_err_mutex;
int32_t* g_err_ptr[kMaxDevices] = {};

int32_t* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mutex);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int32_t*>(p);
  }
  return g_err_ptr[dev];
}

std::mutex g_stage_mutex;
kda::Stages g_stages = {};

kda::Stages current_stages() {
  std::lock_guard<std::mutex> lock(g_stage_mutex);
  return g_stages;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t elem_size(int32_t dt) { return dt == KDA_DTYPE_BF16 ? 2 : 4; }

// Checks shared by prefill and decode; fills the launch record's sizes.
kda_status_t check_common(const kda_params_t* p, Problem* P) {
  if (!p) return KDA_ERR_INVALID_ARG;
  if (p->num_seqs < 0 || p->num_k_heads <= 0 || p->num_v_heads <= 0 || p->num_slots <= 0)
    return KDA_ERR_INVALID_ARG;
  if (p->num_v_heads % p->num_k_heads != 0) return KDA_ERR_INVALID_ARG;
  if (p->num_v_heads > 65535) return KDA_ERR_UNSUPPORTED;
  if (p->d_k != p->d_v) return KDA_ERR_UNSUPPORTED;
  if (p->d_k != 16 && p->d_k != 128) return KDA_ERR_UNSUPPORTED;
  if (p->qkv_dtype != KDA_DTYPE_F32 && p->qkv_dtype != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARG;
  if (p->state_dtype != KDA_DTYPE_F32 && p->state_dtype != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARG;
  if (p->decay_kind != KDA_DECAY_SCALAR && p->decay_kind != KDA_DECAY_PER_CHANNEL)
    return KDA_ERR_INVALID_ARG;
  if (p->flags & ~(KDA_FLAG_CHECKED | KDA_FLAG_CUDA_CORES | KDA_FLAG_COMPACT | KDA_FLAG_NO_DELTA))
    return KDA_ERR_INVALID_ARG;
  const int64_t es = static_cast<int64_t>(elem_size(p->qkv_dtype));
  const int64_t dq = static_cast<int64_t>(p->num_k_heads) * p->d_k;
  const int64_t dv = static_cast<int64_t>(p->num_v_heads) * p->d_v;
  const int64_t qs = p->q_row_stride ? p->q_row_stride : dq;
  const int64_t ks = p->k_row_stride ? p->k_row_stride : dq;
  const int64_t vs = p->v_row_stride ? p->v_row_stride : dv;
  if (qs < dq || ks < dq || vs < dv) return KDA_ERR_INVALID_ARG;
  if ((qs * es) % 16 || (ks * es) % 16 || (vs * es) % 16) return KDA_ERR_INVALID_ARG;
  P->num_seqs = p->num_seqs;
  P->HK = p->num_k_heads;
  P->HV = p->num_v_heads;
  P->D = p->d_k;
  P->num_slots = p->num_slots;
  P->chunk = p->chunk;
  P->T = p->total_tokens;
  P->scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf(static_cast<float>(p->d_k));
  P->l2norm = p->l2norm_qk ? 1 : 0;
  P->flags = p->flags;
  P->q_stride = qs;
  P->k_stride = ks;
  P->v_stride = vs;
  return KDA_OK;
}

kda_status_t check_prefill(const kda_params_t* p, Problem* P) {
  kda_status_t s = check_common(p, P);
  if (s != KDA_OK) return s;
  if (p->total_tokens < 0 || p->total_tokens > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (p->chunk != 16 && p->chunk != 32 && p->chunk != 64) return KDA_ERR_UNSUPPORTED;
  if (p->num_seqs > 0x3fffffff) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

kda_status_t to_status(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

// The tensor-core path serves bf16 inputs at d = 128, chunk 64 unless the caller
// asks for CUDA cores; everything else runs the fp32 CUDA-core path.
bool use_tc(const kda_params_t* p, const Problem& P) {
  return !(p->flags & KDA_FLAG_CUDA_CORES) &&
         kda::tc_prefill_supported(P, p->qkv_dtype == KDA_DTYPE_BF16);
}

// Tensor-core path: by default a chunk-parallel front kernel writes every chunk's chain
// operands to the workspace and a chain kernel walks each sequence; KDA_FLAG_COMPACT runs
// both parts in one kernel per (sequence, head, value tile) with only the chunk table.
bool compact_tc(const kda_params_t* p) { return (p->flags & KDA_FLAG_COMPACT) != 0; }

size_t prefill_workspace_bytes(const kda_params_t* p, const Problem& P) {
  if (!use_tc(p, P)) return kda::simt_workspace_bytes(P);
  return compact_tc(p) ? kda::tc_workspace_bytes(P) : kda::split_workspace_bytes(P);
}

// The prefill path chosen for p, on a fully filled-in Problem.
kda_status_t prefill_dispatch(const kda_params_t* p, const Problem& P, void* workspace, cudaStream_t stream) {
  const bool qbf16 = p->qkv_dtype == KDA_DTYPE_BF16;
  const bool sbf16 = p->state_dtype == KDA_DTYPE_BF16;
  const bool perch = p->decay_kind == KDA_DECAY_PER_CHANNEL;
  const kda::Stages st = current_stages();
  if (use_tc(p, P)) {
    if (compact_tc(p)) return to_status(kda::launch_prefill_tc(P, workspace, perch, sbf16, stream, st));
    return to_status(kda::launch_prefill_split(P, workspace, perch, sbf16, stream, st));
  }
  return to_status(kda::launch_prefill_simt(P, workspace, qbf16, perch, sbf16, stream, st));
}

// Gated DeltaProduct: the parameters of the virtual sequence (n_h positions per token, dense
// virtual queries; k and v keep the caller's stride between substep rows).  For the decode
// form (one token per sequence) total_tokens is num_seqs and a chunk of 0 means 64.
constexpr int32_t kMaxSubsteps = 64;
kda_status_t gdp_virtual_params(const kda_params_t* p, int32_t n_h, bool decode, kda_params_t* pv) {
  if (!p || n_h < 1 || n_h > kMaxSubsteps) return KDA_ERR_INVALID_ARG;
  if (p->flags & KDA_FLAG_NO_DELTA) return KDA_ERR_UNSUPPORTED;   // defined on the delta rule
  *pv = *p;
  const int64_t T = decode ? static_cast<int64_t>(p->num_seqs) : p->total_tokens;
  if (T < 0) return KDA_ERR_INVALID_ARG;
  if (T * n_h > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
  pv->total_tokens = T * n_h;
  pv->q_row_stride = 0;
  if (decode && pv->chunk == 0) pv->chunk = 64;
  return KDA_OK;
}

// Workspace of the GDP forms: [virtual offsets | virtual q | virtual log-decay | virtual o |
// the prefill's own workspace], 256-byte aligned pieces.
struct GdpLayout {
  size_t offv, qv, gv, ov, inner, total;
};
GdpLayout gdp_layout(const kda_params_t* pv, const Problem& Pv) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t Tv = static_cast<size_t>(Pv.T);
  const size_t es = elem_size(pv->qkv_dtype);
  const size_t gw = pv->decay_kind == KDA_DECAY_PER_CHANNEL ? static_cast<size_t>(Pv.D) : 1;
  GdpLayout L;
  L.offv = 0;
  L.qv = up(L.offv + (static_cast<size_t>(Pv.num_seqs) + 1) * 4);
  L.gv = up(L.qv + Tv * Pv.HK * Pv.D * es);
  L.ov = up(L.gv + Tv * Pv.HV * gw * 4);
  L.inner = up(L.ov + Tv * Pv.HV * Pv.D * 4);
  L.total = L.inner + prefill_workspace_bytes(pv, Pv);
  return L;
}

kda_status_t gdp_run(const kda_params_t* p, int32_t n_h, bool decode, const void* q, const void* k,
                     const void* v, const float* beta, const float* log_decay,
                     const uint32_t* input_row_offsets, const uint32_t* slot_idx, void* state_pool,
                     float* o, void* workspace, size_t workspace_bytes, void* stream) {
  kda_params_t pv;
  kda_status_t s = gdp_virtual_params(p, n_h, decode, &pv);
  if (s != KDA_OK) return s;
  Problem P{};
  s = check_prefill(&pv, &P);
  if (s != KDA_OK) return s;
  if (p->num_seqs == 0) return KDA_OK;
  if ((!decode && !input_row_offsets) || !slot_idx || !state_pool) return KDA_ERR_INVALID_ARG;
  if (P.T > 0 && (!q || !k || !v || !beta || !log_decay || !o)) return KDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(state_pool, 16) || !aligned(beta, 4) || !aligned(log_decay, 4) ||
      !aligned(input_row_offsets, 4) || !aligned(slot_idx, 4))
    return KDA_ERR_INVALID_ARG;
  // the caller's query rows (one per token) keep its stride
  const int64_t dq = static_cast<int64_t>(p->num_k_heads) * p->d_k;
  const int64_t q_stride = p->q_row_stride ? p->q_row_stride : dq;
  if (q_stride < dq || (q_stride * static_cast<int64_t>(elem_size(p->qkv_dtype))) % 16) return KDA_ERR_INVALID_ARG;
  const GdpLayout L = gdp_layout(&pv, P);
  if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256)) return KDA_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  uint32_t* offv = reinterpret_cast<uint32_t*>(ws + L.offv);
  void* qv = ws + L.qv;
  float* gv = reinterpret_cast<float*>(ws + L.gv);
  float* ov = reinterpret_cast<float*>(ws + L.ov);
  const int64_t T = P.T / n_h;
  const int64_t grow = static_cast<int64_t>(P.HV) * (p->decay_kind == KDA_DECAY_PER_CHANNEL ? P.D : 1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (to_status(kda::launch_gdp_expand(q, q_stride, p->qkv_dtype == KDA_DTYPE_BF16, log_decay,
                                       decode ? nullptr : input_row_offsets, T, n_h, dq, grow,
                                       p->num_seqs, qv, gv, offv, st)) != KDA_OK)
    return KDA_ERR_CUDA;
  P.q = qv; P.k = k; P.v = v; P.beta = beta; P.g = gv;
  P.offsets = offv; P.slot_idx = slot_idx;
  P.pool = state_pool; P.o = ov;
  P.err = device_error_word();
  if (!P.err) return KDA_ERR_CUDA;
  s = prefill_dispatch(&pv, P, ws + L.inner, st);
  if (s != KDA_OK) return s;
  return to_status(kda::launch_gdp_gather(ov, T, n_h, static_cast<int64_t>(P.HV) * P.D, o, st));
}

}  // namespace

extern "C" {

int kda_abi_version(void) { return KDA_ABI_VERSION; }

const char* kda_status_string(kda_status_t s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

int kda_prefill_uses_tensor_cores(const kda_params_t* p) {
  Problem P{};
  if (check_prefill(p, &P) != KDA_OK) return -1;
  return use_tc(p, P) ? 1 : 0;
}

kda_status_t kda_prefill_workspace_size(const kda_params_t* p, size_t* bytes) {
  Problem P{};
  if (!bytes) return KDA_ERR_INVALID_ARG;
  kda_status_t s = check_prefill(p, &P);
  if (s != KDA_OK) return s;
  *bytes = prefill_workspace_bytes(p, P);
  return KDA_OK;
}

kda_status_t kda_prefill_fwd(const kda_params_t* p, const void* q, const void* k, const void* v,
                             const float* beta, const float* log_decay,
                             const uint32_t* input_row_offsets, const uint32_t* slot_idx,
                             void* state_pool, float* o, void* workspace, size_t workspace_bytes,
                             void* stream) {
  Problem P{};
  kda_status_t s = check_prefill(p, &P);
  if (s != KDA_OK) return s;
  if (p->num_seqs == 0) return KDA_OK;
  if (!input_row_offsets || !slot_idx || !state_pool) return KDA_ERR_INVALID_ARG;
  if (p->total_tokens > 0 && (!q || !k || !v || !beta || !log_decay || !o)) return KDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(state_pool, 16) || !aligned(beta, 4) || !aligned(log_decay, 4) ||
      !aligned(input_row_offsets, 4) || !aligned(slot_idx, 4))
    return KDA_ERR_INVALID_ARG;
  // per-channel log-decay rows are staged in 16-byte pieces (tensor copies, cp.async)
  if (p->decay_kind == KDA_DECAY_PER_CHANNEL && !aligned(log_decay, 16)) return KDA_ERR_INVALID_ARG;
  const size_t need = prefill_workspace_bytes(p, P);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return KDA_ERR_WORKSPACE;
  P.q = q; P.k = k; P.v = v; P.beta = beta; P.g = log_decay;
  P.offsets = input_row_offsets; P.slot_idx = slot_idx;
  P.pool = state_pool; P.o = o;
  P.err = device_error_word();
  if (!P.err) return KDA_ERR_CUDA;
  return prefill_dispatch(p, P, workspace, static_cast<cudaStream_t>(stream));
}

kda_status_t kda_prefill_bwd_workspace_size(const kda_params_t* p, size_t* bytes) {
  Problem P{};
  if (!bytes) return KDA_ERR_INVALID_ARG;
  kda_status_t s = check_prefill(p, &P);
  if (s != KDA_OK) return s;
  *bytes = kda::bwd_workspace_bytes(P, p->qkv_dtype == KDA_DTYPE_BF16, (p->flags & KDA_FLAG_COMPACT) != 0);
  return KDA_OK;
}

kda_status_t kda_prefill_bwd(const kda_params_t* p, const void* q, const void* k, const void* v,
                             const float* beta, const float* log_decay,
                             const uint32_t* input_row_offsets, const uint32_t* slot_idx,
                             const void* state_pool, const float* d_o, const float* d_state,
                             float* dq, float* dk, float* dv, float* dbeta, float* dlog_decay,
                             float* d_state0, void* workspace, size_t workspace_bytes,
                             void* stream) {
  Problem P{};
  kda_status_t s = check_prefill(p, &P);
  if (s != KDA_OK) return s;
  if (p->num_seqs == 0) return KDA_OK;
  if (!input_row_offsets || !slot_idx || !state_pool) return KDA_ERR_INVALID_ARG;
  if (p->total_tokens > 0 && (!q || !k || !v || !beta || !log_decay || !d_o || !dq || !dk ||
                              !dv || !dbeta || !dlog_decay))
    return KDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(state_pool, 4) ||
      !aligned(beta, 4) || !aligned(log_decay, 4) || !aligned(input_row_offsets, 4) ||
      !aligned(slot_idx, 4) || !aligned(d_o, 4) || !aligned(d_state, 4) || !aligned(dq, 4) ||
      !aligned(dk, 4) || !aligned(dv, 4) || !aligned(dbeta, 4) || !aligned(dlog_decay, 4) ||
      !aligned(d_state0, 4))
    return KDA_ERR_INVALID_ARG;
  const size_t need = kda::bwd_workspace_bytes(P, p->qkv_dtype == KDA_DTYPE_BF16, (p->flags & KDA_FLAG_COMPACT) != 0);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return KDA_ERR_WORKSPACE;
  P.q = q; P.k = k; P.v = v; P.beta = beta; P.g = log_decay;
  P.offsets = input_row_offsets; P.slot_idx = slot_idx;
  P.pool = const_cast<void*>(state_pool);   // read only: the initial states
  P.o = nullptr;
  P.err = device_error_word();
  if (!P.err) return KDA_ERR_CUDA;
  return to_status(kda::launch_prefill_bwd(
      P, workspace, d_o, d_state, dq, dk, dv, dbeta, dlog_decay, d_state0,
      p->qkv_dtype == KDA_DTYPE_BF16, p->decay_kind == KDA_DECAY_PER_CHANNEL,
      p->state_dtype == KDA_DTYPE_BF16, (p->flags & KDA_FLAG_COMPACT) != 0,
      static_cast<cudaStream_t>(stream)));
}

kda_status_t kda_conv_gates_fwd(const kda_params_t* p, int32_t width, const void* x,
                                const float* conv_weight, const float* conv_bias, const float* a,
                                const float* b, const float* A_log, const float* dt_bias,
                                const uint32_t* input_row_offsets, const uint32_t* slot_idx,
                                void* conv_state, void* y, float* log_decay, float* beta,
                                void* stream) {
  Problem P{};
  kda_status_t s = check_common(p, &P);
  if (s != KDA_OK) return s;
  if (width < 1 || width > 4) return KDA_ERR_UNSUPPORTED;
  if (p->q_row_stride || p->k_row_stride || p->v_row_stride) return KDA_ERR_INVALID_ARG;
  // without offsets every sequence is one token (the decode form)
  const int64_t T = input_row_offsets ? p->total_tokens : p->num_seqs;
  if (T < 0 || T > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (p->num_seqs == 0 || T == 0) return KDA_OK;
  if (!conv_weight || !x || !y || !a || !b || !log_decay || !beta) return KDA_ERR_INVALID_ARG;
  if (conv_state && width > 1 && !slot_idx) return KDA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(conv_state, 4) || !aligned(conv_weight, 4) ||
      !aligned(conv_bias, 4) || !aligned(a, 4) || !aligned(b, 4) || !aligned(A_log, 4) ||
      !aligned(dt_bias, 4) || !aligned(input_row_offsets, 4) || !aligned(slot_idx, 4) ||
      !aligned(log_decay, 4) || !aligned(beta, 4))
    return KDA_ERR_INVALID_ARG;
  const int CD = 2 * p->num_k_heads * p->d_k + p->num_v_heads * p->d_v;
  const int GW = p->decay_kind == KDA_DECAY_PER_CHANNEL ? p->d_k : 1;
  int32_t* err = device_error_word();
  if (!err) return KDA_ERR_CUDA;
  return to_status(kda::launch_conv_gates(
      x, conv_weight, conv_bias, a, b, A_log, dt_bias, input_row_offsets, slot_idx,
      width > 1 ? conv_state : nullptr, y, log_decay, beta, T, p->num_seqs, CD, p->num_v_heads,
      GW, p->num_slots, width, p->qkv_dtype == KDA_DTYPE_BF16, err,
      static_cast<cudaStream_t>(stream)));
}

kda_status_t kda_gdp_workspace_size(const kda_params_t* p, int32_t n_h, int32_t decode, size_t* bytes) {
  if (!bytes) return KDA_ERR_INVALID_ARG;
  kda_params_t pv;
  kda_status_t s = gdp_virtual_params(p, n_h, decode != 0, &pv);
  if (s != KDA_OK) return s;
  Problem P{};
  s = check_prefill(&pv, &P);
  if (s != KDA_OK) return s;
  *bytes = gdp_layout(&pv, P).total;
  return KDA_OK;
}

kda_status_t kda_gdp_prefill_fwd(const kda_params_t* p, int32_t n_h, const void* q, const void* k,
                                 const void* v, const float* beta, const float* log_decay,
                                 const uint32_t* input_row_offsets, const uint32_t* slot_idx,
                                 void* state_pool, float* o, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  return gdp_run(p, n_h, false, q, k, v, beta, log_decay, input_row_offsets, slot_idx, state_pool,
                 o, workspace, workspace_bytes, stream);
}

kda_status_t kda_gdp_decode_step(const kda_params_t* p, int32_t n_h, const void* q, const void* k,
                                 const void* v, const float* beta, const float* log_decay,
                                 const uint32_t* slot_idx, void* state_pool, float* o,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  return gdp_run(p, n_h, true, q, k, v, beta, log_decay, nullptr, slot_idx, state_pool, o,
                 workspace, workspace_bytes, stream);
}

kda_status_t kda_decode_step(const kda_params_t* p, const void* q, const void* k, const void* v,
                             const float* beta, const float* log_decay, const uint32_t* slot_idx,
                             void* state_pool, float* o, void* stream) {
  Problem P{};
  kda_status_t s = check_common(p, &P);
  if (s != KDA_OK) return s;
  if (p->num_seqs == 0) return KDA_OK;
  if (static_cast<int64_t>(p->num_seqs) * p->num_v_heads > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !beta || !log_decay || !slot_idx || !state_pool || !o) return KDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(state_pool, 16) || !aligned(beta, 4) || !aligned(log_decay, 4) || !aligned(slot_idx, 4))
    return KDA_ERR_INVALID_ARG;
  P.T = p->num_seqs;
  P.q = q; P.k = k; P.v = v; P.beta = beta; P.g = log_decay;
  P.slot_idx = slot_idx; P.pool = state_pool; P.o = o;
  P.err = device_error_word();
  if (!P.err) return KDA_ERR_CUDA;
  const kda::Stages st = current_stages();
  return to_status(kda::launch_decode(P, p->qkv_dtype == KDA_DTYPE_BF16,
                                      p->state_dtype == KDA_DTYPE_BF16,
                                      p->decay_kind == KDA_DECAY_PER_CHANNEL,
                                      static_cast<cudaStream_t>(stream), st));
}

int kda_ring_record_elems(const kda_params_t* p) {
  Problem P{};
  if (check_common(p, &P) != KDA_OK) return -1;
  return kda::ring_record_elems(P.D, p->decay_kind == KDA_DECAY_PER_CHANNEL);
}

kda_status_t kda_verify_window(const kda_params_t* p, const void* q, const void* k, const void* v,
                               const float* beta, const float* log_decay, const uint32_t* slot_idx,
                               int32_t window, const void* state_pool, float* o, float* ring,
                               void* stream) {
  Problem P{};
  kda_status_t s = check_common(p, &P);
  if (s != KDA_OK) return s;
  if (window < 1 || window > 64) return KDA_ERR_INVALID_ARG;
  if (p->num_seqs == 0) return KDA_OK;
  if (static_cast<int64_t>(p->num_seqs) * p->num_v_heads > 0x7fffffffLL ||
      static_cast<int64_t>(p->num_seqs) * window > 0x7fffffffLL)
    return KDA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !beta || !log_decay || !slot_idx || !state_pool || !o || !ring)
    return KDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(state_pool, 16) || !aligned(ring, 16) || !aligned(beta, 4) ||
      !aligned(log_decay, 4) || !aligned(slot_idx, 4))
    return KDA_ERR_INVALID_ARG;
  P.T = static_cast<int64_t>(p->num_seqs) * window;
  P.q = q; P.k = k; P.v = v; P.beta = beta; P.g = log_decay;
  P.slot_idx = slot_idx; P.pool = const_cast<void*>(state_pool); P.o = o;
  P.err = device_error_word();
  if (!P.err) return KDA_ERR_CUDA;
  return to_status(kda::launch_verify(P, window, ring, p->qkv_dtype == KDA_DTYPE_BF16,
                                      p->state_dtype == KDA_DTYPE_BF16,
                                      p->decay_kind == KDA_DECAY_PER_CHANNEL,
                                      static_cast<cudaStream_t>(stream)));
}

kda_status_t kda_fold_accepted(const kda_params_t* p, const float* ring, int32_t window,
                               const uint32_t* accepted, const uint32_t* slot_idx,
                               void* state_pool, void* stream) {
  Problem P{};
  kda_status_t s = check_common(p, &P);
  if (s != KDA_OK) return s;
  if (window < 1 || window > 64) return KDA_ERR_INVALID_ARG;
  if (p->num_seqs == 0) return KDA_OK;
  if (static_cast<int64_t>(p->num_seqs) * p->num_v_heads > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
  if (!ring || !accepted || !slot_idx || !state_pool) return KDA_ERR_INVALID_ARG;
  if (!aligned(ring, 16) || !aligned(state_pool, 16) || !aligned(accepted, 4) ||
      !aligned(slot_idx, 4))
    return KDA_ERR_INVALID_ARG;
  P.slot_idx = slot_idx;
  P.pool = state_pool;
  P.err = device_error_word();
  if (!P.err) return KDA_ERR_CUDA;
  return to_status(kda::launch_fold(P, window, ring, accepted, p->state_dtype == KDA_DTYPE_BF16,
                                    p->decay_kind == KDA_DECAY_PER_CHANNEL,
                                    static_cast<cudaStream_t>(stream)));
}

kda_status_t kda_get_device_error(void* stream, int32_t* code) {
  if (!code) return KDA_ERR_INVALID_ARG;
  int32_t* w = device_error_word();
  if (!w) return KDA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_CUDA;
  int32_t val = 0;
  if (cudaMemcpy(&val, w, sizeof(val), cudaMemcpyDeviceToHost) != cudaSuccess) return KDA_ERR_CUDA;
  if (val != 0) {
    const int32_t zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return KDA_ERR_CUDA;
  }
  *code = val;
  return val ? KDA_ERR_DEVICE : KDA_OK;
}

kda_status_t kda_set_stage_events(void* const* events, int32_t count) {
  if (count < 0 || count > 8) return KDA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_stage_mutex);
  g_stages.n = events ? count : 0;
  for (int i = 0; i < g_stages.n; ++i) g_stages.ev[i] = static_cast<cudaEvent_t>(events[i]);
  return KDA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Prefill without device allocation: the scratch is this file-scope array.
// Host code must not pass the array's name to a kernel (on the host it names a
// stand-in, not device memory); its device address is looked up once per device
// with cudaGetSymbolAddress and cached.
static __device__ __align__(256) unsigned char g_kda_no_alloc_scratch[KDA_NO_ALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_no_alloc_mutex;
void* g_no_alloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (nullptr on failure).
void* no_alloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_no_alloc_mutex);
  if (!g_no_alloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_kda_no_alloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_no_alloc_ptr[dev] = ptr;
  }
  return g_no_alloc_ptr[dev];
}
}  // namespace

namespace {
// The parameters kda_prefill_fwd_no_alloc runs: the two-kernel tensor-core form when its
// chunk records fit the scratch, else the compact form.  False when nothing fits.
bool no_alloc_params(const kda_params_t* p, const Problem& P, kda_params_t* q_params) {
  *q_params = *p;
  if (use_tc(p, P) && prefill_workspace_bytes(p, P) > KDA_NO_ALLOC_SCRATCH_BYTES)
    q_params->flags |= KDA_FLAG_COMPACT;
  return prefill_workspace_bytes(q_params, P) <= KDA_NO_ALLOC_SCRATCH_BYTES;
}
}  // namespace

extern "C" int kda_prefill_no_alloc_form(const kda_params_t* p) {
  Problem P{};
  if (check_prefill(p, &P) != KDA_OK) return -1;
  kda_params_t q_params;
  if (!no_alloc_params(p, P, &q_params)) return -1;
  if (!use_tc(&q_params, P)) return 2;
  return compact_tc(&q_params) ? 1 : 0;
}

extern "C" kda_status_t kda_prefill_fwd_no_alloc(const kda_params_t* p, const void* q,
                                                 const void* k, const void* v,
                                                 const float* beta, const float* log_decay,
                                                 const uint32_t* input_row_offsets,
                                                 const uint32_t* slot_idx, void* state_pool,
                                                 float* o, void* stream) {
  Problem P{};
  kda_status_t s = check_prefill(p, &P);
  if (s != KDA_OK) return s;
  // the tensor-core path falls back to its single-kernel form when the chunk records
  // of the two-kernel form do not fit the scratch
  kda_params_t q_params;
  if (!no_alloc_params(p, P, &q_params)) return KDA_ERR_WORKSPACE;
  if (p->num_seqs == 0) return KDA_OK;
  void* scratch = no_alloc_scratch();
  if (!scratch) return KDA_ERR_CUDA;
  return kda_prefill_fwd(&q_params, q, k, v, beta, log_decay, input_row_offsets, slot_idx,
                         state_pool, o, scratch, KDA_NO_ALLOC_SCRATCH_BYTES, stream);
}
