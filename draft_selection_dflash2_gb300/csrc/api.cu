// api.cu -- the C ABI of libdflash2: handle management, host-side argument
// validation and dispatch to the kernels.  The handle owns one device buffer,
// the 4-byte error word; every other byte a call needs is the caller's.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "dflash2.h"
#include "common.cuh"
#include "launch.h"

struct dflash2_handle {
  int device = 0;
  int num_sms = 0;
  uint32_t* err = nullptr;      // device error word
};

namespace {

constexpr int kK = 16;
constexpr int64_t kMaxL = 64;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA; }

// Launch errors are sticky per thread in the runtime; surface them as a status.
int launched(cudaError_t e) {
  if (e != cudaSuccess) return DFLASH2_ERR_CUDA;
  return from_cuda(cudaGetLastError());
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

bool bad_handle(const dflash2_handle* h) { return h == nullptr || h->err == nullptr; }

// Kernels launch on the calling thread's current device and write the handle's
// error word, which lives on the handle's device: a call made while another
// device is current is refused before anything launches.
int wrong_device(const dflash2_handle* h) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH2_ERR_CUDA;
  return dev == h->device ? DFLASH2_OK : DFLASH2_ERR_INVALID_ARG;
}

// One NVTX range per compute call, named after the entry point, so a timeline
// (Nsight Systems, or any NVTX tool) shows the library's calls; without a tool
// attached a push/pop costs a few nanoseconds.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace

extern "C" {

int dflash2_version(void) { return 100; }

const char* dflash2_status_string(int status) {
  switch (status) {
    case DFLASH2_OK: return "ok";
    case DFLASH2_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH2_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case DFLASH2_ERR_MISALIGNED: return "misaligned pointer or leading dimension";
    case DFLASH2_ERR_CUDA: return "CUDA runtime error";
    case DFLASH2_ERR_TIMEOUT: return "bounded device wait timed out";
    case DFLASH2_ERR_DEVICE: return "device reported an error";
    case DFLASH2_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int dflash2_create(int device, dflash2_handle** out) {
  if (out == nullptr) return DFLASH2_ERR_INVALID_ARG;
  *out = nullptr;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count)
    return DFLASH2_ERR_INVALID_ARG;
  if (cudaSetDevice(device) != cudaSuccess) return DFLASH2_ERR_CUDA;
  dflash2_handle* h = new (std::nothrow) dflash2_handle;
  if (h == nullptr) return DFLASH2_ERR_CUDA;
  h->device = device;
  if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaMalloc(&h->err, sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(h->err, 0, sizeof(uint32_t)) != cudaSuccess) {
    if (h->err) cudaFree(h->err);
    delete h;
    return DFLASH2_ERR_CUDA;
  }
  *out = h;
  return DFLASH2_OK;
}

int dflash2_destroy(dflash2_handle* h) {
  if (h == nullptr) return DFLASH2_ERR_INVALID_ARG;
  int st = DFLASH2_OK;
  if (h->err) {
    if (cudaSetDevice(h->device) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
      st = DFLASH2_ERR_CUDA;
    cudaFree(h->err);
  }
  delete h;
  return st;
}

int dflash2_num_sms(const dflash2_handle* h) { return h ? h->num_sms : 0; }

int dflash2_get_device_error(dflash2_handle* h, void* stream, uint32_t* bits, int clear) {
  if (bad_handle(h) || bits == nullptr) return DFLASH2_ERR_INVALID_ARG;
  if (const int st = wrong_device(h)) return st;
  cudaStream_t s = as_stream(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DFLASH2_ERR_CUDA;
  if (cudaMemcpy(bits, h->err, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DFLASH2_ERR_CUDA;
  if (clear && cudaMemset(h->err, 0, sizeof(uint32_t)) != cudaSuccess) return DFLASH2_ERR_CUDA;
  return DFLASH2_OK;
}

int dflash2_topk(dflash2_handle* h, const uint16_t* logits, int64_t rows, int64_t V, int64_t ld,
                 int k, float* vals, int32_t* idx, void* stream) {
  const NvtxRange range("dflash2_topk");
  if (bad_handle(h) || rows < 0 || V < 0 || ld < V) return DFLASH2_ERR_INVALID_ARG;
  if (k != kK || V < kK || V >= (int64_t(1) << 31)) return DFLASH2_ERR_UNSUPPORTED;
  if (rows == 0) return DFLASH2_OK;
  if (!logits || !vals || !idx) return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(logits, 16) || (ld % 8) != 0 || !aligned(vals, 4) || !aligned(idx, 4))
    return DFLASH2_ERR_MISALIGNED;
  if (const int st = wrong_device(h)) return st;
  // gridDim.y is limited to 65535 rows per launch
  for (int64_t r0 = 0; r0 < rows; r0 += 65535) {
    const int64_t n = rows - r0 < 65535 ? rows - r0 : 65535;
    const int st = launched(dflash2::launch_topk(logits + r0 * ld, n, V, ld, vals + r0 * kK,
                                                 idx + r0 * kK, h->err, h->num_sms, as_stream(stream)));
    if (st != DFLASH2_OK) return st;
  }
  return DFLASH2_OK;
}

size_t dflash2_pair_scores_workspace(const dflash2_handle* h, int64_t B, int64_t L, int64_t d) {
  if (bad_handle(h) || B <= 0 || L <= 0 || d <= 0 || d % 64 != 0) return 0;
  return dflash2::gate_workspace_bytes(B, L, d, h->num_sms);
}

int dflash2_pair_scores(dflash2_handle* h, const int32_t* cand_idx, const float* cand_val,
                        const int32_t* last_verified, const uint16_t* hs, const uint16_t* W_H,
                        const float* b_H, const uint16_t* A, const uint16_t* Bt, int64_t B,
                        int64_t L, int64_t d, int64_t V, float* gate, float* S, void* workspace,
                        size_t ws_bytes, void* stream) {
  const NvtxRange range("dflash2_pair_scores");
  if (bad_handle(h) || B < 0 || L < 0 || d <= 0 || V <= 0) return DFLASH2_ERR_INVALID_ARG;
  if (L > kMaxL || d % 64 != 0 || V >= (int64_t(1) << 31)) return DFLASH2_ERR_UNSUPPORTED;
  if (B == 0 || L == 0) return DFLASH2_OK;
  if (!cand_idx || !cand_val || !last_verified || !hs || !W_H || !A || !Bt || !gate || !S)
    return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(hs, 16) || !aligned(W_H, 16) || !aligned(A, 16) || !aligned(Bt, 16) ||
      !aligned(gate, 16) || !aligned(S, 16) || !aligned(cand_idx, 4) || !aligned(cand_val, 4) ||
      !aligned(last_verified, 4) || (b_H && !aligned(b_H, 4)) || (workspace && !aligned(workspace, 256)))
    return DFLASH2_ERR_MISALIGNED;
  if (workspace == nullptr || ws_bytes < dflash2::gate_workspace_bytes(B, L, d, h->num_sms))
    return DFLASH2_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  if (const int st = wrong_device(h)) return st;
  const int st = launched(dflash2::launch_gate(hs, W_H, b_H, B * L, d, gate, workspace, h->err, h->num_sms, s));
  if (st != DFLASH2_OK) return st;
  return launched(dflash2::launch_pair_scores(cand_idx, cand_val, last_verified, static_cast<const float*>(workspace),
                                              b_H, gate, d, A, Bt, B, L, V, S, h->err, h->num_sms, s));
}

int dflash2_walk(dflash2_handle* h, const float* S, const int32_t* cand_idx, int64_t B, int64_t L,
                 float temperature, uint64_t seed, uint64_t offset, int32_t* draft_tok,
                 int32_t* draft_slot, float* draft_q, void* stream) {
  const NvtxRange range("dflash2_walk");
  if (bad_handle(h) || B < 0 || L < 0) return DFLASH2_ERR_INVALID_ARG;
  if (L > kMaxL || B >= (int64_t(1) << 31)) return DFLASH2_ERR_UNSUPPORTED;
  if (!(temperature == temperature)) return DFLASH2_ERR_INVALID_ARG;   // NaN
  if (B == 0 || L == 0) return DFLASH2_OK;
  if (!S || !cand_idx || !draft_tok || !draft_slot) return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(S, 16) || !aligned(cand_idx, 4) || !aligned(draft_tok, 4) || !aligned(draft_slot, 4) ||
      (draft_q && !aligned(draft_q, 4)))
    return DFLASH2_ERR_MISALIGNED;
  if (const int st = wrong_device(h)) return st;
  return launched(dflash2::launch_walk(S, cand_idx, B, L, temperature, seed, offset, draft_tok,
                                       draft_slot, draft_q, h->err, as_stream(stream)));
}

int dflash2_walk_viterbi(dflash2_handle* h, const float* S, const int32_t* cand_idx, int64_t B, int64_t L,
                         int32_t* draft_tok, int32_t* draft_slot, float* score, void* stream) {
  const NvtxRange range("dflash2_walk_viterbi");
  if (bad_handle(h) || B < 0 || L < 0) return DFLASH2_ERR_INVALID_ARG;
  if (L > kMaxL || B >= (int64_t(1) << 31)) return DFLASH2_ERR_UNSUPPORTED;
  if (B == 0 || L == 0) return DFLASH2_OK;
  if (!S || !cand_idx || !draft_tok || !draft_slot) return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(S, 16) || !aligned(cand_idx, 4) || !aligned(draft_tok, 4) || !aligned(draft_slot, 4) ||
      (score && !aligned(score, 4)))
    return DFLASH2_ERR_MISALIGNED;
  if (const int st = wrong_device(h)) return st;
  return launched(dflash2::launch_walk_viterbi(S, cand_idx, B, L, draft_tok, draft_slot, score, h->err,
                                                   as_stream(stream)));
}

int dflash2_selector_eval(dflash2_handle* h, const int32_t* gt, const int32_t* cand_idx, int64_t B, int64_t L,
                          int32_t* accept1, int32_t* accept16, int64_t* counts, void* stream) {
  const NvtxRange range("dflash2_selector_eval");
  if (bad_handle(h) || B < 0 || L < 0) return DFLASH2_ERR_INVALID_ARG;
  if (L > kMaxL || B >= (int64_t(1) << 31)) return DFLASH2_ERR_UNSUPPORTED;
  if (L == 0) return DFLASH2_OK;
  if (!counts || (B > 0 && (!gt || !cand_idx || !accept1 || !accept16))) return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(counts, 8) || (B > 0 && (!aligned(gt, 4) || !aligned(cand_idx, 4) || !aligned(accept1, 4) ||
                                        !aligned(accept16, 4))))
    return DFLASH2_ERR_MISALIGNED;
  if (const int st = wrong_device(h)) return st;
  return launched(dflash2::launch_selector_eval(gt, cand_idx, B, L, accept1, accept16, counts, h->num_sms,
                                                    as_stream(stream)));
}

size_t dflash2_conv2tap_workspace(const dflash2_handle* h, int64_t B, int64_t L, int64_t d) {
  if (bad_handle(h) || B <= 0 || L <= 0 || d <= 0 || d % 64 != 0) return 0;
  return dflash2::conv_workspace_bytes(B, L, d, h->num_sms);
}

int dflash2_conv2tap(dflash2_handle* h, const uint16_t* x, const uint16_t* x_prev,
                     const uint16_t* hs, const uint16_t* k0, const uint16_t* k1,
                     const uint16_t* W_c, const float* b_c, int64_t B, int64_t L, int64_t d,
                     void* y, int y_is_fp32, void* workspace, size_t ws_bytes, void* stream) {
  const NvtxRange range("dflash2_conv2tap");
  if (bad_handle(h) || B < 0 || L < 0 || d <= 0) return DFLASH2_ERR_INVALID_ARG;
  if (d % 64 != 0 || L > kMaxL || B > 65535) return DFLASH2_ERR_UNSUPPORTED;
  if (B == 0 || L == 0) return DFLASH2_OK;
  if (!x || !x_prev || !k0 || !k1 || !W_c || !y) return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(x_prev, 16) || (hs && !aligned(hs, 16)) || !aligned(k0, 16) ||
      !aligned(k1, 16) || !aligned(W_c, 16) || !aligned(y, 16) || (b_c && !aligned(b_c, 4)) ||
      (workspace && !aligned(workspace, 256)))
    return DFLASH2_ERR_MISALIGNED;
  if (workspace == nullptr || ws_bytes < dflash2::conv_workspace_bytes(B, L, d, h->num_sms))
    return DFLASH2_ERR_WORKSPACE;
  if (const int st = wrong_device(h)) return st;
  return launched(dflash2::launch_conv2tap(x, x_prev, hs, k0, k1, W_c, b_c, B, L, d, y, y_is_fp32, workspace,
                                           h->err, h->num_sms, as_stream(stream)));
}

size_t dflash2_gemm_conv2tap_workspace(const dflash2_handle* h, int64_t B, int64_t L, int64_t d) {
  if (bad_handle(h) || B <= 0 || L <= 0 || d <= 0) return 0;
  return dflash2::gemm_conv_workspace_bytes(B, L, d);
}

int dflash2_gemm_conv2tap(dflash2_handle* h, const uint16_t* A, const uint16_t* W, const uint16_t* x_prev,
                          const uint16_t* hs, const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c,
                          const float* b_c, int64_t B, int64_t L, int64_t K, int64_t d, float* c_work,
                          size_t c_bytes, void* y, int y_is_fp32, void* stream) {
  const NvtxRange range("dflash2_gemm_conv2tap");
  if (bad_handle(h) || B < 0 || L < 0 || K <= 0 || d <= 0) return DFLASH2_ERR_INVALID_ARG;
  if (d % 64 != 0 || K % 64 != 0 || L > kMaxL || B * L >= (int64_t(1) << 31)) return DFLASH2_ERR_UNSUPPORTED;
  if (B == 0 || L == 0) return DFLASH2_OK;
  if (!A || !W || !x_prev || !hs || !k0 || !k1 || !W_c || !c_work || !y) return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(W, 16) || !aligned(x_prev, 16) || !aligned(hs, 16) || !aligned(k0, 16) ||
      !aligned(k1, 16) || !aligned(W_c, 16) || !aligned(c_work, 16) || !aligned(y, 16) || (b_c && !aligned(b_c, 4)))
    return DFLASH2_ERR_MISALIGNED;
  if (c_bytes < dflash2::gemm_conv_workspace_bytes(B, L, d)) return DFLASH2_ERR_WORKSPACE;
  if (const int st = wrong_device(h)) return st;
  return launched(dflash2::launch_gemm_conv2tap(A, W, x_prev, hs, k0, k1, W_c, b_c, B, L, K, d, c_work, y, y_is_fp32,
                                                h->err, h->num_sms, as_stream(stream)));
}

size_t dflash2_verify_workspace(const dflash2_handle* h, int64_t B, int64_t L, int64_t V) {
  if (bad_handle(h) || B <= 0 || L < 0 || L > kMaxL || V <= 0 || V > dflash2::verify_max_vocab()) return 0;
  return dflash2::verify_workspace_bytes(B, L, V);
}

int dflash2_verify(dflash2_handle* h, const uint16_t* target, int64_t ld, const int32_t* draft_tok,
                   const int32_t* draft_slot, const float* draft_q, const int32_t* cand_idx,
                   int64_t B, int64_t L, int64_t V, float temperature, uint64_t seed,
                   uint64_t offset, int32_t* accept_len, int32_t* out_tok, void* workspace,
                   size_t ws_bytes, void* stream) {
  const NvtxRange range("dflash2_verify");
  if (bad_handle(h) || B < 0 || L < 0 || V <= 0 || ld < V) return DFLASH2_ERR_INVALID_ARG;
  if (L > kMaxL || V > dflash2::verify_max_vocab()) return DFLASH2_ERR_UNSUPPORTED;
  if (!(temperature == temperature)) return DFLASH2_ERR_INVALID_ARG;
  if (B == 0) return DFLASH2_OK;
  const bool sampled = temperature > 0.0f;
  // an empty block (L = 0) reads no draft: only the bonus row is decided
  if (!target || (L > 0 && !draft_tok) || !accept_len || !out_tok) return DFLASH2_ERR_INVALID_ARG;
  if (sampled && L > 0 && (!draft_slot || !draft_q || !cand_idx)) return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(target, 16) || (ld % 8) != 0 || !aligned(draft_tok, 4) || !aligned(accept_len, 4) ||
      !aligned(out_tok, 4) || (draft_slot && !aligned(draft_slot, 4)) ||
      (draft_q && !aligned(draft_q, 4)) || (cand_idx && !aligned(cand_idx, 4)) ||
      (workspace && !aligned(workspace, 256)))
    return DFLASH2_ERR_MISALIGNED;
  if (workspace == nullptr || ws_bytes < dflash2::verify_workspace_bytes(B, L, V)) return DFLASH2_ERR_WORKSPACE;
  if (const int st = wrong_device(h)) return st;
  return launched(dflash2::launch_verify(target, ld, draft_tok, draft_slot, draft_q, cand_idx, B, L, V,
                                         temperature, seed, offset, accept_len, out_tok, workspace, h->err,
                                         h->num_sms, as_stream(stream)));
}

size_t dflash2_lmhead_topk_workspace(const dflash2_handle* h, int64_t M, int64_t V, int64_t d) {
  if (bad_handle(h) || M <= 0 || V <= 0 || d <= 0) return 0;
  return dflash2::lmhead_workspace_bytes(M, V, d, h->num_sms);
}

int dflash2_lmhead_topk(dflash2_handle* h, const uint16_t* hidden, const uint16_t* W, int64_t M,
                        int64_t V, int64_t d, float* vals, int32_t* idx, void* workspace,
                        size_t ws_bytes, void* stream) {
  const NvtxRange range("dflash2_lmhead_topk");
  if (bad_handle(h) || M < 0 || V < 0 || d <= 0) return DFLASH2_ERR_INVALID_ARG;
  if (d % 64 != 0 || V < kK || V >= (int64_t(1) << 31)) return DFLASH2_ERR_UNSUPPORTED;
  if (M == 0) return DFLASH2_OK;
  if (!hidden || !W || !vals || !idx) return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(vals, 4) || !aligned(idx, 4) ||
      (workspace && !aligned(workspace, 256)))
    return DFLASH2_ERR_MISALIGNED;
  if (workspace == nullptr || ws_bytes < dflash2::lmhead_workspace_bytes(M, V, d, h->num_sms))
    return DFLASH2_ERR_WORKSPACE;
  if (const int st = wrong_device(h)) return st;
  return launched(dflash2::launch_lmhead_topk(hidden, W, M, V, d, vals, idx, workspace, h->num_sms,
                                              h->err, as_stream(stream)));
}

int dflash2_lmhead_topk_gate(dflash2_handle* h, const uint16_t* hidden, const uint16_t* W, const uint16_t* W_H,
                             const float* b_H, int64_t M, int64_t V, int64_t d, float* vals, int32_t* idx,
                             float* gate, void* workspace, size_t ws_bytes, void* stream) {
  const NvtxRange range("dflash2_lmhead_topk_gate");
  if (bad_handle(h) || M < 0 || V < 0 || d <= 0) return DFLASH2_ERR_INVALID_ARG;
  if (d % 64 != 0 || V < kK || V >= (int64_t(1) << 31) - 256) return DFLASH2_ERR_UNSUPPORTED;
  if (M == 0) return DFLASH2_OK;
  if (!hidden || !W || !W_H || !vals || !idx || !gate) return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(W_H, 16) || !aligned(vals, 4) || !aligned(idx, 4) ||
      !aligned(gate, 16) || (b_H && !aligned(b_H, 4)) || (workspace && !aligned(workspace, 256)))
    return DFLASH2_ERR_MISALIGNED;
  if (workspace == nullptr || ws_bytes < dflash2::lmhead_workspace_bytes(M, V, d, h->num_sms))
    return DFLASH2_ERR_WORKSPACE;
  if (const int st = wrong_device(h)) return st;
  return launched(dflash2::launch_lmhead_topk_gate(hidden, W, W_H, b_H, M, V, d, vals, idx, gate, workspace,
                                                   h->num_sms, h->err, as_stream(stream)));
}

size_t dflash2_pair_scores_proj_workspace(const dflash2_handle* h, int64_t B, int64_t L) {
  if (bad_handle(h) || B <= 0 || L <= 0 || L > kMaxL) return 0;
  return dflash2::proj_workspace_bytes(B, L);
}

int dflash2_pair_scores_proj(dflash2_handle* h, const int32_t* cand_idx, const float* cand_val,
                             const int32_t* last_verified, const float* gate, const uint16_t* E,
                             const uint16_t* W_A, const uint16_t* W_B, int64_t B, int64_t L, int64_t d, int64_t V,
                             float* P, size_t P_bytes, float* S, void* stream) {
  const NvtxRange range("dflash2_pair_scores_proj");
  if (bad_handle(h) || B < 0 || L < 0 || d <= 0 || V <= 0) return DFLASH2_ERR_INVALID_ARG;
  if (d % 64 != 0 || L > kMaxL || V >= (int64_t(1) << 31) || B * L >= (int64_t(1) << 26))
    return DFLASH2_ERR_UNSUPPORTED;
  if (B == 0 || L == 0) return DFLASH2_OK;
  if (!cand_idx || !cand_val || !last_verified || !gate || !E || !W_A || !W_B || !P || !S)
    return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(cand_idx, 4) || !aligned(cand_val, 4) || !aligned(last_verified, 4) || !aligned(gate, 16) ||
      !aligned(E, 16) || !aligned(W_A, 16) || !aligned(W_B, 16) || !aligned(P, 16) || !aligned(S, 4))
    return DFLASH2_ERR_MISALIGNED;
  if (P_bytes < dflash2::proj_workspace_bytes(B, L)) return DFLASH2_ERR_WORKSPACE;
  if (const int st = wrong_device(h)) return st;
  return launched(dflash2::launch_pair_scores_proj(cand_idx, cand_val, last_verified, gate, E, W_A, W_B, B, L, d,
                                                   V, P, S, h->num_sms, h->err, as_stream(stream)));
}

int dflash2_selftest_wait_timeout(dflash2_handle* h, uint64_t limit_ns, uint32_t* words, void* stream) {
  const NvtxRange range("dflash2_selftest_wait_timeout");
  if (bad_handle(h) || words == nullptr || limit_ns == 0 || limit_ns > dflash2::kWaitLimitNs)
    return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(words, 4)) return DFLASH2_ERR_MISALIGNED;
  if (const int st = wrong_device(h)) return st;
  return launched(dflash2::launch_wait_timeout_selftest(words, limit_ns, h->err, words + 1, as_stream(stream)));
}

int dflash2_lmhead_topk_noalloc(dflash2_handle* h, const uint16_t* hidden, const uint16_t* W, int64_t M,
                                int64_t V, int64_t d, float* vals, int32_t* idx, void* stream) {
  const NvtxRange range("dflash2_lmhead_topk_noalloc");
  if (bad_handle(h) || M < 0 || V < 0 || d <= 0) return DFLASH2_ERR_INVALID_ARG;
  if (d % 64 != 0 || V < kK || V >= (int64_t(1) << 31)) return DFLASH2_ERR_UNSUPPORTED;
  if (M == 0) return DFLASH2_OK;
  if (!hidden || !W || !vals || !idx) return DFLASH2_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(vals, 4) || !aligned(idx, 4))
    return DFLASH2_ERR_MISALIGNED;
  if (dflash2::lmhead_workspace_bytes(M, V, d, h->num_sms) > dflash2::kLmheadNoAllocScratchBytes)
    return DFLASH2_ERR_WORKSPACE;
  if (const int st = wrong_device(h)) return st;
  void* scratch = nullptr;
  if (dflash2::lmhead_noalloc_scratch(h->device, &scratch) != cudaSuccess) return DFLASH2_ERR_CUDA;
  return launched(dflash2::launch_lmhead_topk(hidden, W, M, V, d, vals, idx, scratch, h->num_sms, h->err,
                                              as_stream(stream)));
}

}  // extern "C"
