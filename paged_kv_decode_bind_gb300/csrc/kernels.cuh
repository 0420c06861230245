// Internal launch interface between the C-ABI layer (pkv_api.cu) and the
// kernel translation units.  Every launcher returns cudaGetLastError().
#pragma once

#include "common.cuh"

namespace pkv {

cudaError_t launch_bind_meta(const pkv_workspace &ws, int batch, int mode, cudaStream_t st);
cudaError_t launch_flat_index(const pkv_workspace &ws, int batch, cudaStream_t st);
cudaError_t launch_append(const pkv_workspace &ws, int batch, int layer_begin, int layer_count,
                          const void *k_new, const void *v_new, cudaStream_t st);
int meta_max_batch();

struct DecodeArgs {
  pkv_workspace ws;
  int batch;
  int layer;
  const void *q;
  float scale;
  int num_splits;
  int flags;
  const void *k_new;  // fused append source (bf16 [batch, Hkv, D]) or NULL
  const void *v_new;
  int fused_merge;    // 1: the last split of each (request, KV head) merges
  int apportion;      // tensor-core kernel: apportioned splits (set by its launcher)
};

// CUDA-core split-KV decode.  Returns cudaErrorNotSupported for shapes
// without an instantiation.
cudaError_t launch_decode_simt(const DecodeArgs &a, cudaStream_t st);
bool decode_simt_supported(int head_dim, int group);

// Tensor-core (warp mma) split-KV decode; same contract as the SIMT kernel,
// plus the fused append and merge.
cudaError_t launch_decode_mma(const DecodeArgs &a, cudaStream_t st);
// The step's split plan for the tensor-core kernel (pkv_plan_step) and the
// size of ws.work_plan it needs.
cudaError_t launch_plan(const DecodeArgs &a, cudaStream_t st);
size_t plan_bytes();
bool decode_mma_supported(int head_dim, int group);

cudaError_t launch_merge(const pkv_workspace &ws, int batch, int num_splits, int flags,
                         cudaStream_t st);

}  // namespace pkv
