// launch.h -- internal kernel launchers behind the C ABI (not exported).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "dflash2.h"

namespace dflash2 {

constexpr int kMaxDevices = 64;

// Kernel attributes are per device: these set one for the current device the
// first time a launch there needs it.  One record per kernel (Fn) and device.
// A launch attribute that lets the kernel start while the previous kernel in
// the stream finishes; the kernel calls pdl_wait before its first global access.
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a = {};
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

template <auto Fn>
cudaError_t set_smem_limit(size_t bytes) {
  static std::mutex mu;
  static size_t done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(Fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done[dev] = bytes;
  return e;
}

template <auto Fn>
cudaError_t allow_nonportable_clusters() {
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(Fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

int topk_cluster_size(int64_t rows, int64_t V, int num_sms);
cudaError_t launch_topk(const uint16_t* logits, int64_t rows, int64_t V, int64_t ld, float* vals,
                        int32_t* idx, uint32_t* err, int num_sms, cudaStream_t stream);

// The gate contraction's split-K partials ([ks, B*L, 256] fp32) go to the
// workspace (the pair kernel turns them into H).
size_t gate_workspace_bytes(int64_t B, int64_t L, int64_t d, int num_sms);
cudaError_t launch_gate(const uint16_t* hs, const uint16_t* W_H, const float* b_H, int64_t M,
                        int64_t d, float* gate, void* workspace, uint32_t* err, int num_sms, cudaStream_t stream);
// The pair scores; the gate H is formed here from the gate GEMM's partials
// (gate_part, as launch_gate left them) and written to `gate`.
cudaError_t launch_pair_scores(const int32_t* cand_idx, const float* cand_val,
                               const int32_t* last_verified, const float* gate_part, const float* b_H, float* gate,
                               int64_t d, const uint16_t* A, const uint16_t* Bt, int64_t B, int64_t L, int64_t V,
                               float* S, uint32_t* err, int num_sms, cudaStream_t stream);

cudaError_t launch_walk(const float* S, const int32_t* cand_idx, int64_t B, int64_t L,
                        float temperature, uint64_t seed, uint64_t offset, int32_t* draft_tok,
                        int32_t* draft_slot, float* draft_q, uint32_t* err, cudaStream_t stream);

// The two-tap conv (conv2tap.cu): the correction's split-K partials go to the
// workspace ([ks, B*L, 2d/16] fp32), then the taps.
size_t conv_workspace_bytes(int64_t B, int64_t L, int64_t d, int num_sms);
cudaError_t launch_conv2tap(const uint16_t* x, const uint16_t* x_prev, const uint16_t* hs,
                            const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c,
                            const float* b_c, int64_t B, int64_t L, int64_t d, void* y,
                            int y_is_fp32, void* workspace, uint32_t* err, int num_sms, cudaStream_t stream);

cudaError_t launch_walk_viterbi(const float* S, const int32_t* cand_idx, int64_t B, int64_t L, int32_t* draft_tok,
                                int32_t* draft_slot, float* score, uint32_t* err, cudaStream_t stream);

cudaError_t launch_selector_eval(const int32_t* gt, const int32_t* cand_idx, int64_t B, int64_t L, int32_t* accept1,
                                 int32_t* accept16, int64_t* counts, int num_sms, cudaStream_t stream);

// Device workspace (barrier words, per-row arrival counters, row maxima and
// sums, per-chunk sums) that launch_verify needs for B sequences of L
// positions over a V-id vocabulary, at either temperature.
size_t verify_workspace_bytes(int64_t B, int64_t L, int64_t V);
// Largest vocabulary launch_verify handles (10,485,760 ids).
int64_t verify_max_vocab();

cudaError_t launch_verify(const uint16_t* target, int64_t ld, const int32_t* draft_tok,
                          const int32_t* draft_slot, const float* draft_q, const int32_t* cand_idx,
                          int64_t B, int64_t L, int64_t V, float temperature, uint64_t seed,
                          uint64_t offset, int32_t* accept_len, int32_t* out_tok, void* workspace,
                          uint32_t* err, int num_sms, cudaStream_t stream);

size_t lmhead_workspace_bytes(int64_t M, int64_t V, int64_t d, int num_sms);
cudaError_t launch_lmhead_topk_gate(const uint16_t* hidden, const uint16_t* W, const uint16_t* W_H,
                                    const float* b_H, int64_t M, int64_t V, int64_t d, float* vals, int32_t* idx,
                                    float* gate, void* workspace, int num_sms, uint32_t* err, cudaStream_t stream);

// The two-tap conv fused into its producing GEMM (gemm_conv.cu): c = W_c h +
// b_c into c_work ([B*L, 2d/16] fp32), then y = taps(A W^T).
size_t gemm_conv_workspace_bytes(int64_t B, int64_t L, int64_t d);
cudaError_t launch_gemm_conv2tap(const uint16_t* A, const uint16_t* W, const uint16_t* x_prev, const uint16_t* hs,
                                 const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c, const float* b_c,
                                 int64_t B, int64_t L, int64_t K, int64_t d, float* c_work, void* y, int y_is_fp32,
                                 uint32_t* err, int num_sms, cudaStream_t stream);

// Projection-form pair scores: P = [W_A E(id); W_B E(id)] for the step's
// candidates and last verified tokens, then S from P (proj.cu).
size_t proj_rows(int64_t B, int64_t L);
size_t proj_workspace_bytes(int64_t B, int64_t L);
cudaError_t launch_pair_scores_proj(const int32_t* cand_idx, const float* cand_val, const int32_t* last_verified,
                                    const float* gate, const uint16_t* E, const uint16_t* W_A, const uint16_t* W_B,
                                    int64_t B, int64_t L, int64_t d, int64_t V, float* P, float* S, int num_sms,
                                    uint32_t* err, cudaStream_t stream);
// A kernel whose two bounded waits (an mbarrier, a global word) cannot be
// satisfied; each gives up after limit_ns (selftest.cu).
cudaError_t launch_wait_timeout_selftest(const uint32_t* flag, uint64_t limit_ns, uint32_t* err, uint32_t* result,
                                         cudaStream_t stream);

constexpr size_t kLmheadNoAllocScratchBytes = DFLASH2_LMHEAD_NOALLOC_SCRATCH_BYTES;
cudaError_t lmhead_noalloc_scratch(int device, void** ptr);
cudaError_t launch_lmhead_topk(const uint16_t* hidden, const uint16_t* W, int64_t M, int64_t V,
                               int64_t d, float* vals, int32_t* idx, void* workspace,
                               int num_sms, uint32_t* err, cudaStream_t stream);

}  // namespace dflash2
