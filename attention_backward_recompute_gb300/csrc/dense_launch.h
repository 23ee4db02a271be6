// Host-side launchers of the dense kernels (called from api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "dense_common.cuh"

namespace attn {

// TMA descriptors of one dense call.  Q-like tensors (q, dy) and K-like tensors
// (k, v) are described twice, with boxes of 64 and 128 rows (64 columns each,
// 128-byte swizzle); the bias tensor [B,H,Sq,Sk] with boxes of 64 keys x 64 or
// 128 queries.
struct DenseMaps {
  CUtensorMap q64, q128, dy64, dy128;
  CUtensorMap k64, k128, v64, v128;
  CUtensorMap bias64, bias128;
  // fp32 storage: the maps above address the hi copies (bf16) of the split
  // inputs and these the lo copies; without split they repeat the maps above.
  CUtensorMap q64_lo, q128_lo, dy64_lo, dy128_lo;
  CUtensorMap k64_lo, k128_lo, v64_lo, v128_lo;
  bool split;
};

// padded head dim handled by the tensor-core kernels: 64 or 128
inline int padded_head_dim(int D) { return D <= 64 ? 64 : 128; }

cudaError_t launch_fwd_stats(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s);
// bf16 storage: row statistics from S and dP (no O accumulator), Q and dY in tensor memory
cudaError_t launch_stats2(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s);
// x[0, n) = value
cudaError_t launch_fill_f32(float* x, float value, int64_t n, cudaStream_t s);
// per-element mask [BH, Sq, Sk] fp32 -> row and column bit sets (see DenseParams)
cudaError_t launch_pack_elem_mask(const float* m, float thr, int64_t BH, int Sq, int Sk, uint32_t* rows,
                                  uint32_t* cols, int ew_q, int ew_k, cudaStream_t s);
// zero the D elements (es bytes each) of every (b, s, h) row of a strided tensor
cudaError_t launch_zero_rows(void* x, int64_t sb, int64_t ss, int64_t sh, int64_t B, int64_t S, int64_t H, int64_t D,
                             size_t es, cudaStream_t s);
cudaError_t launch_delta_only(const DenseParams& p, int dtype_bf16, cudaStream_t s);
// Split fp32 tensors into hi/lo bf16 copies: hi = bf16(x), lo = bf16(x - hi).
// hi = bf16(x), lo = bf16(x - hi) for up to four fp32 tensors of n[i]
// elements (multiples of 4; a count <= 0 skips the tensor), one launch.
cudaError_t launch_split_f32(const float* const x[4], void* const hi[4], void* const lo[4], const int64_t n[4],
                             cudaStream_t s);
cudaError_t launch_dkdv(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s);
// bf16 storage: softmax and dS on separate warpgroups, P and dS in tensor memory
cudaError_t launch_dkdv2(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s);
cudaError_t launch_dq(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s);
// bf16 storage: softmax and dS on separate warpgroups, P and dS in tensor memory
cudaError_t launch_dq2(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s);
// bf16 storage with p.ds_store: dQ = scale * dS K from the dS tiles the dK/dV kernel stored
cudaError_t launch_dq3(const DenseMaps& m, const DenseParams& p, cudaStream_t s);

}  // namespace attn
