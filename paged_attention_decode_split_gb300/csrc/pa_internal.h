// pa_internal.h -- host-side interfaces between the C-ABI layer and the
// translation units that instantiate the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "decode_mma.cuh"
#include "decode_split.cuh"
#include "verify_tc.cuh"

namespace pa {

// Kernel variants compiled into the library; returns false for (D, G) pairs
// outside the set (the C ABI then answers PA_ERR_UNSUPPORTED).
bool decode_supported(int head_dim, int group);
bool verify_supported(int head_dim, int rows);  // rows = q_len * G

// Launch helpers; they return the launch error (cudaSuccess if queued).
cudaError_t launch_decode(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeParams &p, dim3 grid, cudaStream_t stream);
cudaError_t launch_decode_fp8(int head_dim, int group, const CUtensorMap &tk, const CUtensorMap &tv,
                              const DecodeParams &p, dim3 grid, cudaStream_t stream);
cudaError_t launch_reduce(int head_dim, const ReduceParams &p, int rows, int num_sms, cudaStream_t stream);
// Whether a bf16 verify of this shape runs 128-key score tiles (it then reads
// K through tk128, whole 128-token tiles of one page).
bool verify_wide_score_tiles(int head_dim, int rows);
cudaError_t launch_verify(int head_dim, int rows, const CUtensorMap &tk, const CUtensorMap &tv,
                          const CUtensorMap &tk64, const CUtensorMap &tv64, const CUtensorMap &tk128,
                          const VerifyParams &p, dim3 grid, cudaStream_t stream);

cudaError_t launch_verify_fp8(int head_dim, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tk64,
                              const CUtensorMap &tv64, const VerifyParams &p, dim3 grid, cudaStream_t stream);

// Sets the dynamic shared-memory limit of `fn` once per device.
cudaError_t ensure_smem_limit(const void *fn, int bytes, int slot);

}  // namespace pa
