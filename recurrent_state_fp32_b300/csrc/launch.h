// Internal launcher interface between the C ABI (api.cu) and the kernel files.
// Arguments are validated by the caller; launchers only pick tile shapes,
// grids and template instances.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "replayssm.h"

namespace rs {

// Layout of state.work: rows of `row` floats per (sequence, draft, head) --
// Mamba-2: buffer terms [0, P) and decay at P; delta: swept query [0, d_k)
// and buffer terms [d_k, d_k + d_v) -- then one int32 flag per sequence.
struct WorkLayout {
  int row;         // floats per row (a multiple of 4)
  long long rows;  // batch * K * heads
  long long batch;
  WorkLayout(const replayssm_dims& d, int K) {
    const int need = d.kind == REPLAYSSM_MAMBA2 ? d.dv + 1 : d.dk + d.dv;
    row = (need + 3) & ~3;
    batch = d.batch;
    rows = batch * (K < 1 ? 1 : K) * d.heads;
  }
  long long bytes() const { return rows * row * 4 + ((batch * 4 + 15) & ~15LL); }
  int32_t* flags(float* work) const { return reinterpret_cast<int32_t*>(work + rows * row); }
};

// Entries a fused fold + decode step folds at most (W <= kStepMaxW).
constexpr int kStepMaxW = 16;

// Layout of state.work for the fused Mamba-2 fold + decode step: one row of
// kStepRow floats per (sequence, head) -- the decode weights
// c_j = w_j (C . B_j) of the buffered entries at [0, kStepMaxW) (zero past
// the entries the decode replays), the token's weight plus D at kStepTok,
// the decode decay at kStepDecay, the fold decay at kStepFoldDecay and the
// fold weights w_j at [kStepFoldW, kStepFoldW + kStepMaxW) -- then per
// (sequence, group) the folded B rows as [kStepMaxW][N] floats.
constexpr int kStepTok = kStepMaxW;
constexpr int kStepDecay = kStepMaxW + 1;
constexpr int kStepFoldDecay = kStepMaxW + 2;
constexpr int kStepFoldW = kStepMaxW + 4;
constexpr int kStepRow = kStepFoldW + kStepMaxW;
struct StepLayout {
  long long rows, bf0, total;  // float offsets
  explicit StepLayout(const replayssm_dims& d) {
    rows = (long long)d.batch * d.heads;
    bf0 = rows * kStepRow;
    total = bf0 + (long long)d.batch * d.groups * kStepMaxW * d.dk;
  }
  long long bytes() const { return total * 4; }
};

// Device facts cached per device (SM count, opt-in shared memory per block).
struct DeviceInfo {
  int sms;
  int smem_optin;  // shared memory one block may opt in to
  int smem_sm;     // shared memory per SM, all resident blocks together
};
const DeviceInfo& device_info();

cudaError_t launch_mamba2_decode(const replayssm_dims& d, const replayssm_state& s, const float* A,
                                 const float* D, const void* x, const void* B, const void* C,
                                 const float* dt, float* y, cudaStream_t st);
cudaError_t launch_mamba2_verify(const replayssm_dims& d, const replayssm_state& s, int K,
                                 const float* A, const float* D, const void* x, const void* B,
                                 const void* C, const float* dt, float* y, cudaStream_t st);
cudaError_t launch_mamba2_fold(const replayssm_dims& d, const replayssm_state& s, const float* A,
                               int k_next, int force, cudaStream_t st);
// consolidate(k_next = 1) then decode, as one prep and one stream launch
cudaError_t launch_mamba2_fold_decode(const replayssm_dims& d, const replayssm_state& s,
                                      const float* A, const float* D, const void* x,
                                      const void* B, const void* C, const float* dt, float* y,
                                      cudaStream_t st);
cudaError_t launch_mamba2_conventional(const replayssm_dims& d, float* S, const float* A,
                                       const float* D, const void* x, const void* B, const void* C,
                                       const float* dt, float* y, cudaStream_t st);

cudaError_t launch_delta_decode(const replayssm_dims& d, const replayssm_state& s, const void* q,
                                const void* k, const void* v, const float* alpha,
                                const float* beta, float scale, float* o, cudaStream_t st);
cudaError_t launch_delta_verify(const replayssm_dims& d, const replayssm_state& s, int K,
                                const void* q, const void* k, const void* v, const float* alpha,
                                const float* beta, float scale, float* o, cudaStream_t st);
// Shared memory the fused delta decode / verify block needs at least.
size_t delta_fused_smem(const replayssm_dims& d, int K, bool read16);
// The delta kernel's launch configuration for these sizes (no CUDA call);
// false if none fits in optin bytes of shared memory per block.
bool delta_kernel_config(const replayssm_dims& d, int K, bool read16, size_t optin,
                         replayssm_delta_config& out);
cudaError_t launch_delta_fold(const replayssm_dims& d, const replayssm_state& s, int k_next,
                              int force, cudaStream_t st);
// consolidate(k_next = 1) then decode: the decode grid, then the fold grid
// that folds the full rings and decodes their token from the new rows
cudaError_t launch_delta_fold_decode(const replayssm_dims& d, const replayssm_state& s,
                                     const void* q, const void* k, const void* v,
                                     const float* alpha, const float* beta, float scale, float* o,
                                     cudaStream_t st);
cudaError_t launch_delta_conventional(const replayssm_dims& d, float* S, const void* q,
                                      const void* k, const void* v, const float* alpha,
                                      const float* beta, float scale, float* o, cudaStream_t st);

cudaError_t launch_delta_conventional_verify(const replayssm_dims& d, const float* S, int K,
                                             const void* q, const void* k, const void* v,
                                             const float* alpha, const float* beta, float scale,
                                             float* snap, float* o, cudaStream_t st);
cudaError_t launch_conventional_accept(const replayssm_dims& d, float* S, const float* snap,
                                       const int32_t* m, int K, int32_t* status, cudaStream_t st);

cudaError_t launch_accept(const replayssm_dims& d, const replayssm_state& s, const int32_t* m,
                          int K, cudaStream_t st);
cudaError_t launch_copy_rows(const void* src, void* dst, long long n_bytes, const int32_t* src_idx,
                             const int32_t* dst_idx, int n, int batch, cudaStream_t st);
cudaError_t launch_copy_pointers(const replayssm_state* src, const replayssm_state* dst,
                                 const int32_t* src_idx, const int32_t* dst_idx, int n, int batch,
                                 cudaStream_t st);
cudaError_t launch_refresh(const replayssm_dims& d, const replayssm_state& s, cudaStream_t st);

// Grid for the fold kernels: every block examines at most kFoldTilesPerBlock
// tiles, so its pre-scan of the ring pointers is a single parallel load.
constexpr int kFoldTilesPerBlock = 128;
int fold_grid(long long tiles);

}  // namespace rs
