// C ABI of the ReplaySSM library: host-side argument validation, dispatch to
// the kernel launchers, and the two small kernels (accept, read-copy refresh).
// Argument errors return before any CUDA call; nothing allocates or syncs.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "replayssm.h"

namespace rs {

const DeviceInfo& device_info() {
  static DeviceInfo info[64];
  static std::once_flag once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  std::call_once(once[dev], [dev] {
    int sms = 0, optin = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 148;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      optin = 227 * 1024;
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
        cudaSuccess)
      per_sm = 228 * 1024;
    info[dev] = DeviceInfo{sms, optin, per_sm};
  });
  return info[dev];
}

int fold_grid(long long tiles) {
  const long long min_blocks = (tiles + kMaxFoldTiles - 1) / kMaxFoldTiles;
  const long long want = std::min<long long>(tiles, (long long)device_info().sms * 8);
  return (int)std::max<long long>(std::max(min_blocks, want), 1);
}

namespace {

__global__ void accept_kernel(int batch, int W, int K, const int32_t* __restrict__ m,
                              int32_t* __restrict__ len, int32_t* __restrict__ status) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  const int mv = m[s], l = len[s];
  if (l < 0 || l > W)
    status[s] |= REPLAYSSM_SEQ_BAD_POINTER;
  else if (mv < 0 || mv > K || l + mv > W)
    status[s] |= REPLAYSSM_SEQ_BAD_ACCEPT;
  else
    len[s] = l + mv;
}

// Restores the state of the accepted prefix from its snapshot: block x of
// sequence y copies a slice of snapshot m - 1 into S (m = 0: nothing to do).
__global__ void conventional_accept_kernel(long long per_seq4, int K, const int32_t* __restrict__ m,
                                           const float4* __restrict__ snap,
                                           float4* __restrict__ S, int32_t* __restrict__ status) {
  const int seq = blockIdx.y;
  const int mv = m[seq];
  if (mv < 0 || mv > K) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && status) status[seq] |= REPLAYSSM_SEQ_BAD_ACCEPT;
    return;
  }
  if (mv == 0) return;
  const float4* src = snap + ((long long)seq * K + (mv - 1)) * per_seq4;
  float4* dst = S + (long long)seq * per_seq4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < per_seq4;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// Copies n_bytes (a multiple of 16) per sequence from sequence src_idx[i] of
// src to sequence dst_idx[i] of dst (blockIdx.y = i); pairs with an index
// outside [0, batch) are skipped.
__global__ void copy_rows_kernel(const unsigned char* __restrict__ src, unsigned char* __restrict__ dst,
                                 long long n_bytes, const int32_t* __restrict__ src_idx,
                                 const int32_t* __restrict__ dst_idx, int batch) {
  const int si = src_idx[blockIdx.y], di = dst_idx[blockIdx.y];
  if (si < 0 || si >= batch || di < 0 || di >= batch) return;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + (long long)si * n_bytes);
  uint4* d4 = reinterpret_cast<uint4*>(dst + (long long)di * n_bytes);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_bytes / 16;
       i += (long long)gridDim.x * blockDim.x)
    d4[i] = s4[i];
}

// Per-sequence ring pointers and status of pair i (one thread per pair).
__global__ void copy_pointers_kernel(const int32_t* __restrict__ sh, const int32_t* __restrict__ sl,
                                     const int32_t* __restrict__ ss, int32_t* __restrict__ dh,
                                     int32_t* __restrict__ dl, int32_t* __restrict__ ds,
                                     const int32_t* __restrict__ src_idx,
                                     const int32_t* __restrict__ dst_idx, int n, int batch) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int si = src_idx[i], di = dst_idx[i];
  if (si < 0 || si >= batch || di < 0 || di >= batch) return;
  dh[di] = sh[si];
  dl[di] = sl[si];
  ds[di] = ss[si];
}

// Waits on an mbarrier that nothing arrives at, with the kernels' bounded
// wait: after the limit it records REPLAYSSM_SEQ_TIMEOUT and returns.
__global__ void wait_timeout_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool done = mbar_wait_warp(&bar, 0);
  if (threadIdx.x == 0 && !done) atomicOr(status, REPLAYSSM_SEQ_TIMEOUT);
}

__global__ void refresh_kernel(const float4* __restrict__ S, uint2* __restrict__ R, long long n4) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = S[i];
    R[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

}  // namespace

cudaError_t launch_accept(const replayssm_dims& d, const replayssm_state& s, const int32_t* m,
                          int K, cudaStream_t st) {
  accept_kernel<<<(d.batch + 255) / 256, 256, 0, st>>>(d.batch, d.window, K, m, s.ring_len,
                                                       s.status);
  return cudaGetLastError();
}

cudaError_t launch_conventional_accept(const replayssm_dims& d, float* S, const float* snap,
                                       const int32_t* m, int K, int32_t* status, cudaStream_t st) {
  // one snapshot is H * d_v * d_k floats per sequence (a multiple of 4)
  const long long per_seq4 = (long long)d.heads * d.dv * d.dk / 4;
  const int bx = (int)std::max<long long>(1, std::min<long long>((per_seq4 + 255) / 256, 64));
  conventional_accept_kernel<<<dim3(bx, d.batch), 256, 0, st>>>(
      per_seq4, K, m, reinterpret_cast<const float4*>(snap), reinterpret_cast<float4*>(S), status);
  return cudaGetLastError();
}

cudaError_t launch_copy_rows(const void* src, void* dst, long long n_bytes, const int32_t* src_idx,
                             const int32_t* dst_idx, int n, int batch, cudaStream_t st) {
  const int bx = (int)std::max<long long>(1, std::min<long long>((n_bytes / 16 + 255) / 256, 64));
  copy_rows_kernel<<<dim3(bx, n), 256, 0, st>>>(static_cast<const unsigned char*>(src),
                                                 static_cast<unsigned char*>(dst), n_bytes, src_idx,
                                                 dst_idx, batch);
  return cudaGetLastError();
}

cudaError_t launch_copy_pointers(const replayssm_state* src, const replayssm_state* dst,
                                 const int32_t* src_idx, const int32_t* dst_idx, int n, int batch,
                                 cudaStream_t st) {
  copy_pointers_kernel<<<(n + 255) / 256, 256, 0, st>>>(src->ring_head, src->ring_len, src->status,
                                                        dst->ring_head, dst->ring_len, dst->status,
                                                        src_idx, dst_idx, n, batch);
  return cudaGetLastError();
}

cudaError_t launch_refresh(const replayssm_dims& d, const replayssm_state& s, cudaStream_t st) {
  const long long n4 = (long long)d.batch * d.heads * d.dv * d.dk / 4;
  const long long want = (n4 + 255) / 256;
  const int grid = (int)std::min<long long>(want, (long long)device_info().sms * 16);
  refresh_kernel<<<std::max(grid, 1), 256, 0, st>>>(reinterpret_cast<const float4*>(s.S_ckpt),
                                                    reinterpret_cast<uint2*>(s.S_read), n4);
  return cudaGetLastError();
}

}  // namespace rs

// --------------------------------------------------------------- validation

namespace {

using rs::DeviceInfo;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Null -> INVALID_ARG, misaligned -> MISALIGNED, else OK.
replayssm_status check_ptr(const void* p) {
  if (!p) return REPLAYSSM_ERR_INVALID_ARG;
  return aligned16(p) ? REPLAYSSM_OK : REPLAYSSM_ERR_MISALIGNED;
}

replayssm_status check_opt(const void* p) {
  return (!p || aligned16(p)) ? REPLAYSSM_OK : REPLAYSSM_ERR_MISALIGNED;
}

#define RS_TRY(expr)                               \
  do {                                             \
    const replayssm_status rs_st_ = (expr);        \
    if (rs_st_ != REPLAYSSM_OK) return rs_st_;     \
  } while (0)

replayssm_status check_dims(const replayssm_dims* d) {
  if (!d) return REPLAYSSM_ERR_INVALID_ARG;
  if (d->kind < REPLAYSSM_MAMBA2 || d->kind > REPLAYSSM_KDA) return REPLAYSSM_ERR_INVALID_ARG;
  if (d->batch < 0 || d->heads < 1 || d->groups < 1 || d->dk < 1 || d->dv < 1 || d->window < 1)
    return REPLAYSSM_ERR_INVALID_ARG;
  if (d->in_dtype != REPLAYSSM_F32 && d->in_dtype != REPLAYSSM_BF16)
    return REPLAYSSM_ERR_INVALID_ARG;
  if (d->kind == REPLAYSSM_MAMBA2 && d->heads % d->groups) return REPLAYSSM_ERR_INVALID_ARG;
  if (d->dk != 64 && d->dk != 128) return REPLAYSSM_ERR_UNSUPPORTED;
  if (d->dv % 32 || d->dv > 256) return REPLAYSSM_ERR_UNSUPPORTED;
  if (d->window > 64) return REPLAYSSM_ERR_UNSUPPORTED;
  return REPLAYSSM_OK;
}

replayssm_status check_state(const replayssm_dims* d, const replayssm_state* s) {
  if (!s) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_ptr(s->S_ckpt));
  RS_TRY(check_opt(s->S_read));
  RS_TRY(check_ptr(s->ring_head));
  RS_TRY(check_ptr(s->ring_len));
  RS_TRY(check_ptr(s->status));
  RS_TRY(check_ptr(s->sync));
  RS_TRY(check_ptr(s->work));
  if (d->kind == REPLAYSSM_MAMBA2) {
    RS_TRY(check_ptr(s->ring_x));
    RS_TRY(check_ptr(s->ring_B));
    RS_TRY(check_opt(s->ring_C));
    RS_TRY(check_ptr(s->ring_dt));
  } else {
    RS_TRY(check_opt(s->ring_q));
    RS_TRY(check_ptr(s->ring_k));
    RS_TRY(check_ptr(s->ring_v));
    RS_TRY(check_ptr(s->ring_alpha));
    RS_TRY(check_ptr(s->ring_beta));
  }
  return REPLAYSSM_OK;
}

replayssm_status check_mamba2_token(const void* x, const void* B, const void* C, const float* dt) {
  RS_TRY(check_ptr(x));
  RS_TRY(check_ptr(B));
  RS_TRY(check_ptr(C));
  return check_ptr(dt);
}

replayssm_status check_delta_token(const void* q, const void* k, const void* v,
                                   const float* alpha, const float* beta) {
  RS_TRY(check_ptr(q));
  RS_TRY(check_ptr(k));
  RS_TRY(check_ptr(v));
  RS_TRY(check_ptr(alpha));
  return check_ptr(beta);
}

replayssm_status finish(cudaError_t e) {
  return e == cudaSuccess ? REPLAYSSM_OK : REPLAYSSM_ERR_CUDA;
}

// Shared memory the replay kernels need must fit one block.
replayssm_status check_smem(size_t bytes) {
  return bytes <= (size_t)rs::device_info().smem_optin ? REPLAYSSM_OK : REPLAYSSM_ERR_UNSUPPORTED;
}

}  // namespace

// ------------------------------------------------ fixed scratch (no allocation)

// Scratch of replayssm_mamba2_decode_noalloc: module memory that every device
// loading this library holds until exit; never allocated by a call. Host code
// must not pass the symbol itself to a kernel (on the host it names a
// stand-in, not device memory): it uses the address looked up per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[REPLAYSSM_NOALLOC_SCRATCH_BYTES];

namespace {

// Where the decode scratch lives in the fixed array: the workspace (per-head
// rows, then per-sequence flags), then the per-sequence arrival counters.
struct NoallocLayout {
  long long sync_off, total;
  explicit NoallocLayout(const replayssm_dims& d) {
    sync_off = (rs::WorkLayout(d, 1).bytes() + 255) & ~255LL;
    total = sync_off + 4LL * d.batch;
  }
};

// Device address of g_noalloc_scratch in the current device's context,
// looked up on every call (a cheap query next to the launches): a cached
// address would go stale if the context were torn down and made again.
cudaError_t noalloc_scratch(unsigned char** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<unsigned char*>(p);
  return cudaSuccess;
}

}  // namespace

extern "C" {

REPLAYSSM_API replayssm_status replayssm_mamba2_decode(
    const replayssm_dims* dims, const replayssm_state* state, const float* A, const float* D,
    const void* x, const void* B, const void* C, const float* dt, float* y, void* stream) {
  RS_TRY(check_dims(dims));
  if (dims->kind != REPLAYSSM_MAMBA2) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_state(dims, state));
  RS_TRY(check_ptr(A));
  RS_TRY(check_ptr(D));
  RS_TRY(check_mamba2_token(x, B, C, dt));
  RS_TRY(check_ptr(y));
  if (dims->batch == 0) return REPLAYSSM_OK;
  return finish(rs::launch_mamba2_decode(*dims, *state, A, D, x, B, C, dt, y,
                                         static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_gdn_decode(
    const replayssm_dims* dims, const replayssm_state* state, const void* q, const void* k,
    const void* v, const float* alpha, const float* beta, float scale, float* o, void* stream) {
  RS_TRY(check_dims(dims));
  if (dims->kind == REPLAYSSM_MAMBA2) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_state(dims, state));
  RS_TRY(check_delta_token(q, k, v, alpha, beta));
  RS_TRY(check_ptr(o));
  if (dims->batch == 0) return REPLAYSSM_OK;
  RS_TRY(check_smem(rs::delta_fused_smem(*dims, 1, state->S_read != nullptr)));
  return finish(rs::launch_delta_decode(*dims, *state, q, k, v, alpha, beta, scale, o,
                                        static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_consolidate(const replayssm_dims* dims,
                                                     const replayssm_state* state, const float* A,
                                                     int32_t k_next, int32_t force, void* stream) {
  RS_TRY(check_dims(dims));
  RS_TRY(check_state(dims, state));
  if (k_next < 0 || k_next > dims->window || (force != 0 && force != 1))
    return REPLAYSSM_ERR_INVALID_ARG;
  if (dims->kind == REPLAYSSM_MAMBA2) RS_TRY(check_ptr(A));
  if (dims->batch == 0) return REPLAYSSM_OK;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dims->kind == REPLAYSSM_MAMBA2)
    return finish(rs::launch_mamba2_fold(*dims, *state, A, k_next, force, st));
  return finish(rs::launch_delta_fold(*dims, *state, k_next, force, st));
}

REPLAYSSM_API replayssm_status replayssm_mamba2_fold_decode(
    const replayssm_dims* dims, const replayssm_state* state, const float* A, const float* D,
    const void* x, const void* B, const void* C, const float* dt, float* y, void* stream) {
  RS_TRY(check_dims(dims));
  if (dims->kind != REPLAYSSM_MAMBA2) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_state(dims, state));
  RS_TRY(check_ptr(A));
  RS_TRY(check_ptr(D));
  RS_TRY(check_mamba2_token(x, B, C, dt));
  RS_TRY(check_ptr(y));
  if (dims->batch == 0) return REPLAYSSM_OK;
  return finish(rs::launch_mamba2_fold_decode(*dims, *state, A, D, x, B, C, dt, y,
                                              static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_gdn_fold_decode(
    const replayssm_dims* dims, const replayssm_state* state, const void* q, const void* k,
    const void* v, const float* alpha, const float* beta, float scale, float* o, void* stream) {
  RS_TRY(check_dims(dims));
  if (dims->kind == REPLAYSSM_MAMBA2) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_state(dims, state));
  RS_TRY(check_delta_token(q, k, v, alpha, beta));
  RS_TRY(check_ptr(o));
  if (dims->batch == 0) return REPLAYSSM_OK;
  RS_TRY(check_smem(rs::delta_fused_smem(*dims, 1, state->S_read != nullptr)));
  return finish(rs::launch_delta_fold_decode(*dims, *state, q, k, v, alpha, beta, scale, o,
                                             static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_spec_verify(
    const replayssm_dims* dims, const replayssm_state* state, int32_t K, const void* q,
    const void* k, const void* v, const float* alpha, const float* beta, float scale, float* o,
    void* stream) {
  RS_TRY(check_dims(dims));
  if (dims->kind == REPLAYSSM_MAMBA2) return REPLAYSSM_ERR_UNSUPPORTED;
  if (K < 1 || K > 8) return REPLAYSSM_ERR_INVALID_ARG;
  if (K > dims->window) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_state(dims, state));
  RS_TRY(check_delta_token(q, k, v, alpha, beta));
  RS_TRY(check_ptr(o));
  if (dims->batch == 0) return REPLAYSSM_OK;
  RS_TRY(check_smem(rs::delta_fused_smem(*dims, K, state->S_read != nullptr)));
  return finish(rs::launch_delta_verify(*dims, *state, K, q, k, v, alpha, beta, scale, o,
                                        static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_mamba2_spec_verify(
    const replayssm_dims* dims, const replayssm_state* state, int32_t K, const float* A,
    const float* D, const void* x, const void* B, const void* C, const float* dt, float* y,
    void* stream) {
  RS_TRY(check_dims(dims));
  if (dims->kind != REPLAYSSM_MAMBA2) return REPLAYSSM_ERR_INVALID_ARG;
  if (K < 1 || K > 8 || K > dims->window) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_state(dims, state));
  RS_TRY(check_ptr(A));
  RS_TRY(check_ptr(D));
  RS_TRY(check_mamba2_token(x, B, C, dt));
  RS_TRY(check_ptr(y));
  if (dims->batch == 0) return REPLAYSSM_OK;
  return finish(rs::launch_mamba2_verify(*dims, *state, K, A, D, x, B, C, dt, y,
                                         static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_accept(const replayssm_dims* dims,
                                                const replayssm_state* state, const int32_t* m,
                                                int32_t K, void* stream) {
  RS_TRY(check_dims(dims));
  if (K < 0) return REPLAYSSM_ERR_INVALID_ARG;
  if (!state) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_ptr(state->ring_len));
  RS_TRY(check_ptr(state->status));
  RS_TRY(check_ptr(m));
  if (dims->batch == 0) return REPLAYSSM_OK;
  return finish(rs::launch_accept(*dims, *state, m, K, static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_refresh_read_copy(const replayssm_dims* dims,
                                                           const replayssm_state* state,
                                                           void* stream) {
  RS_TRY(check_dims(dims));
  if (!state) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_ptr(state->S_ckpt));
  RS_TRY(check_ptr(state->S_read));
  if (dims->batch == 0) return REPLAYSSM_OK;
  return finish(rs::launch_refresh(*dims, *state, static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_conventional_mamba2_step(
    const replayssm_dims* dims, float* S, const float* A, const float* D, const void* x,
    const void* B, const void* C, const float* dt, float* y, void* stream) {
  RS_TRY(check_dims(dims));
  if (dims->kind != REPLAYSSM_MAMBA2) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_ptr(S));
  RS_TRY(check_ptr(A));
  RS_TRY(check_ptr(D));
  RS_TRY(check_mamba2_token(x, B, C, dt));
  RS_TRY(check_ptr(y));
  if (dims->batch == 0) return REPLAYSSM_OK;
  return finish(rs::launch_mamba2_conventional(*dims, S, A, D, x, B, C, dt, y,
                                               static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_conventional_gdn_step(
    const replayssm_dims* dims, float* S, const void* q, const void* k, const void* v,
    const float* alpha, const float* beta, float scale, float* o, void* stream) {
  RS_TRY(check_dims(dims));
  if (dims->kind == REPLAYSSM_MAMBA2) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_ptr(S));
  RS_TRY(check_delta_token(q, k, v, alpha, beta));
  RS_TRY(check_ptr(o));
  if (dims->batch == 0) return REPLAYSSM_OK;
  return finish(rs::launch_delta_conventional(*dims, S, q, k, v, alpha, beta, scale, o,
                                              static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_conventional_gdn_verify(
    const replayssm_dims* dims, const float* S, int32_t K, const void* q, const void* k,
    const void* v, const float* alpha, const float* beta, float scale, float* snapshots, float* o,
    void* stream) {
  RS_TRY(check_dims(dims));
  if (dims->kind == REPLAYSSM_MAMBA2) return REPLAYSSM_ERR_INVALID_ARG;
  if (K < 1 || K > 8) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_ptr(S));
  RS_TRY(check_delta_token(q, k, v, alpha, beta));
  RS_TRY(check_ptr(snapshots));
  RS_TRY(check_ptr(o));
  if (dims->batch == 0) return REPLAYSSM_OK;
  return finish(rs::launch_delta_conventional_verify(*dims, S, K, q, k, v, alpha, beta, scale,
                                                     snapshots, o, static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_conventional_accept(const replayssm_dims* dims, float* S,
                                                             const float* snapshots,
                                                             const int32_t* m, int32_t K,
                                                             int32_t* status, void* stream) {
  RS_TRY(check_dims(dims));
  if (K < 1 || K > 8) return REPLAYSSM_ERR_INVALID_ARG;
  RS_TRY(check_ptr(S));
  RS_TRY(check_ptr(snapshots));
  RS_TRY(check_ptr(m));
  RS_TRY(check_opt(status));
  if (dims->batch == 0) return REPLAYSSM_OK;
  if (dims->batch > 65535) return REPLAYSSM_ERR_UNSUPPORTED;
  return finish(rs::launch_conventional_accept(*dims, S, snapshots, m, K, status,
                                               static_cast<cudaStream_t>(stream)));
}

REPLAYSSM_API replayssm_status replayssm_copy_sequences(const replayssm_dims* dims,
                                                       const replayssm_state* src,
                                                       const int32_t* src_idx,
                                                       const replayssm_state* dst,
                                                       const int32_t* dst_idx, int32_t n,
                                                       void* stream) {
  RS_TRY(check_dims(dims));
  RS_TRY(check_state(dims, src));
  RS_TRY(check_state(dims, dst));
  if (n < 0 || n > 65535) return REPLAYSSM_ERR_INVALID_ARG;
  if (n == 0 || dims->batch == 0) return REPLAYSSM_OK;
  RS_TRY(check_ptr(src_idx));
  RS_TRY(check_ptr(dst_idx));
  // optional fields must be present on both sides or on neither
  if (!src->S_read != !dst->S_read) return REPLAYSSM_ERR_INVALID_ARG;
  const bool m2 = dims->kind == REPLAYSSM_MAMBA2;
  if (m2 && !src->ring_C != !dst->ring_C) return REPLAYSSM_ERR_INVALID_ARG;
  if (!m2 && !src->ring_q != !dst->ring_q) return REPLAYSSM_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long H = dims->heads, W = dims->window, Wd = (W + 3) / 4 * 4;
  const long long ti = dims->in_dtype == REPLAYSSM_BF16 ? 2 : 4;
  const long long elems = H * dims->dv * dims->dk;
  const int b = dims->batch;
  cudaError_t e;
#define RS_COPY(SRC, DST, BYTES)                                                           \
  do {                                                                                     \
    e = rs::launch_copy_rows(SRC, DST, BYTES, src_idx, dst_idx, n, b, st);                \
    if (e != cudaSuccess) return REPLAYSSM_ERR_CUDA;                                       \
  } while (0)
  RS_COPY(src->S_ckpt, dst->S_ckpt, elems * 4);
  if (src->S_read) RS_COPY(src->S_read, dst->S_read, elems * 2);
  if (m2) {
    RS_COPY(src->ring_x, dst->ring_x, H * W * dims->dv * ti);
    RS_COPY(src->ring_B, dst->ring_B, W * dims->groups * dims->dk * ti);
    if (src->ring_C) RS_COPY(src->ring_C, dst->ring_C, W * dims->groups * dims->dk * ti);
    RS_COPY(src->ring_dt, dst->ring_dt, H * Wd * 4);
  } else {
    if (src->ring_q) RS_COPY(src->ring_q, dst->ring_q, H * W * dims->dk * ti);
    RS_COPY(src->ring_k, dst->ring_k, H * W * dims->dk * ti);
    RS_COPY(src->ring_v, dst->ring_v, H * W * dims->dv * ti);
    RS_COPY(src->ring_alpha, dst->ring_alpha,
            dims->kind == REPLAYSSM_KDA ? H * W * dims->dk * 4 : H * Wd * 4);
    RS_COPY(src->ring_beta, dst->ring_beta, H * Wd * 4);
  }
#undef RS_COPY
  return finish(rs::launch_copy_pointers(src, dst, src_idx, dst_idx, n, b, st));
}

REPLAYSSM_API replayssm_status replayssm_selftest_wait_timeout(int32_t* status, void* stream) {
  RS_TRY(check_ptr(status));
  rs::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
  return finish(cudaGetLastError());
}

REPLAYSSM_API int64_t replayssm_workspace_bytes(const replayssm_dims* dims, int32_t K) {
  if (check_dims(dims) != REPLAYSSM_OK || K < 0) return 0;
  const long long b = rs::WorkLayout(*dims, K < 1 ? 1 : K).bytes();
  if (dims->kind != REPLAYSSM_MAMBA2) return b;
  return std::max<long long>(b, rs::StepLayout(*dims).bytes());
}

REPLAYSSM_API replayssm_status replayssm_delta_kernel_config(const replayssm_dims* dims,
                                                             int32_t K, int32_t read_copy,
                                                             int64_t smem_limit,
                                                             replayssm_delta_config* out) {
  RS_TRY(check_dims(dims));
  if (!out || dims->kind == REPLAYSSM_MAMBA2 || K < 1 || K > 8 || K > dims->window ||
      smem_limit < 0)
    return REPLAYSSM_ERR_INVALID_ARG;
  const size_t optin = smem_limit ? (size_t)smem_limit : (size_t)232448;
  return rs::delta_kernel_config(*dims, K, read_copy != 0, optin, *out) ? REPLAYSSM_OK
                                                                        : REPLAYSSM_ERR_UNSUPPORTED;
}

REPLAYSSM_API int64_t replayssm_mamba2_decode_noalloc_bytes(const replayssm_dims* dims) {
  if (check_dims(dims) != REPLAYSSM_OK || dims->kind != REPLAYSSM_MAMBA2) return 0;
  return NoallocLayout(*dims).total;
}

REPLAYSSM_API replayssm_status replayssm_mamba2_decode_noalloc(
    const replayssm_dims* dims, const replayssm_state* state, const float* A, const float* D,
    const void* x, const void* B, const void* C, const float* dt, float* y, void* stream) {
  RS_TRY(check_dims(dims));
  if (dims->kind != REPLAYSSM_MAMBA2 || !state) return REPLAYSSM_ERR_INVALID_ARG;
  replayssm_state s = *state;
  // work and sync are replaced by the fixed scratch below: give the pointer
  // checks valid stand-ins for them so that only the caller's fields count.
  s.work = s.S_ckpt;
  s.sync = s.ring_len;
  RS_TRY(check_state(dims, &s));
  RS_TRY(check_ptr(A));
  RS_TRY(check_ptr(D));
  RS_TRY(check_mamba2_token(x, B, C, dt));
  RS_TRY(check_ptr(y));
  const NoallocLayout lay(*dims);
  if (lay.total > (long long)REPLAYSSM_NOALLOC_SCRATCH_BYTES) return REPLAYSSM_ERR_SCRATCH_LIMIT;
  if (dims->batch == 0) return REPLAYSSM_OK;
  unsigned char* base = nullptr;
  if (noalloc_scratch(&base) != cudaSuccess) return REPLAYSSM_ERR_CUDA;
  s.work = reinterpret_cast<float*>(base);
  s.sync = reinterpret_cast<int32_t*>(base + lay.sync_off);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The arrival counters must start at zero; the previous call's contents stay.
  if (cudaMemsetAsync(s.sync, 0, (size_t)dims->batch * 4, st) != cudaSuccess)
    return REPLAYSSM_ERR_CUDA;
  return finish(rs::launch_mamba2_decode(*dims, s, A, D, x, B, C, dt, y, st));
}

REPLAYSSM_API const char* replayssm_status_string(replayssm_status status) {
  switch (status) {
    case REPLAYSSM_OK: return "ok";
    case REPLAYSSM_ERR_INVALID_ARG: return "invalid argument";
    case REPLAYSSM_ERR_UNSUPPORTED: return "unsupported sizes";
    case REPLAYSSM_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case REPLAYSSM_ERR_CUDA: return "CUDA launch error";
    case REPLAYSSM_ERR_SCRATCH_LIMIT:
      return "sizes need more than the 16 MiB fixed scratch of replayssm_mamba2_decode_noalloc";
    default: return "unknown status";
  }
}

REPLAYSSM_API int32_t replayssm_version(void) { return 100; }

}  // extern "C"
