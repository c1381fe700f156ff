// Device helpers shared by the ReplaySSM kernels: bulk copies with mbarrier
// completion (bounded waits), bf16 unpacking, warp reductions, and the
// row-dot engine that streams a state tile from shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "replayssm.h"

namespace rs {

constexpr int kThreads = 128;  // block size of the non-persistent kernels
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;
// Upper bound for any wait on an mbarrier (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// Backstop on the number of polls, in case the timer does not advance.
constexpr uint32_t kWaitLimitPolls = 1u << 26;

typedef __nv_bfloat16 bf16;

// Scalar-per-entry ring fields (Mamba-2 dt, delta beta and GDN alpha) keep
// W entries per (sequence, head) padded to a multiple of 4 floats, so that a
// head's row is a 16-byte multiple and can be bulk-copied.
__host__ __device__ constexpr int ring_wd(int W) { return (W + 3) & ~3; }

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes initialised mbarriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Per-thread asynchronous copies global -> shared (completion: cp_async_wait_all).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch: a grid lets its dependent grid start early,
// and the dependent waits for the full completion (and memory) of the grid
// it depends on before it touches that grid's outputs. Both are no-ops when
// the launch has no programmatic dependency.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk (non-tensor) copy global -> shared; completion counted on `bar` in bytes.
// dst, src and bytes must be multiples of 16. The state stream is read once
// per step, so it is tagged evict-first to leave L2 to the ring.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Same without a cache-policy operand (default L2 behaviour).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes"
      " [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of `bar` to complete; false after ~kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < kWaitLimitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) break;
  }
  return false;
}

// Warp-uniform bounded wait: every lane waits, then the lanes agree, so a
// timeout never splits the warp's control flow.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity)) != 0;
}

// ------------------------------------------------------------ element I/O

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f<bf16>(bf16 v) {
  return __bfloat162float(v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 16 bytes of T as floats: 4 (f32) or 8 (bf16) values.
template <typename T>
struct Chunk {
  static constexpr int kElems = 16 / sizeof(T);
};

template <typename T>
__device__ __forceinline__ void unpack(const uint4 raw, float (&f)[Chunk<T>::kElems]);
template <>
__device__ __forceinline__ void unpack<float>(const uint4 raw, float (&f)[4]) {
  f[0] = __uint_as_float(raw.x);
  f[1] = __uint_as_float(raw.y);
  f[2] = __uint_as_float(raw.z);
  f[3] = __uint_as_float(raw.w);
}
template <>
__device__ __forceinline__ void unpack<bf16>(const uint4 raw, float (&f)[8]) {
  f[0] = bf16_lo(raw.x);
  f[1] = bf16_hi(raw.x);
  f[2] = bf16_lo(raw.y);
  f[3] = bf16_hi(raw.y);
  f[4] = bf16_lo(raw.z);
  f[5] = bf16_hi(raw.z);
  f[6] = bf16_lo(raw.w);
  f[7] = bf16_hi(raw.w);
}

// Two consecutive elements as floats (4- or 8-byte aligned load).
template <typename T>
__device__ __forceinline__ float2 load2(const T* p);
template <>
__device__ __forceinline__ float2 load2<float>(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 load2<bf16>(const bf16* p) {
  const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
  return make_float2(bf16_lo(w), bf16_hi(w));
}

// Round-to-nearest-even pack of two floats into a bf16x2 word (low = a).
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// E consecutive elements of T at p (aligned to E elements) as float, in one
// vector load when E * sizeof(T) is 4, 8 or 16 bytes.
template <typename T, int E>
__device__ __forceinline__ void load_vec(const T* p, float (&out)[E]) {
  constexpr int bytes = E * (int)sizeof(T);
  if constexpr (bytes == 16) {
    unpack<T>(*reinterpret_cast<const uint4*>(p), out);
  } else if constexpr (bytes == 8) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    if constexpr (sizeof(T) == 2) {
      out[0] = bf16_lo(r.x);
      out[1] = bf16_hi(r.x);
      out[2] = bf16_lo(r.y);
      out[3] = bf16_hi(r.y);
    } else {
      out[0] = __uint_as_float(r.x);
      out[1] = __uint_as_float(r.y);
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = to_f(p[e]);
  }
}

// E consecutive elements of T kept as raw 32-bit words (a load that is not
// yet converted holds half the registers for bf16): load_raw issues one
// vector load of E * sizeof(T) bytes (4, 8 or 16), raw_to_f converts.
template <typename T, int E>
struct Raw {
  static constexpr int kWords = (E * (int)sizeof(T) + 3) / 4;
  uint32_t w[kWords];
};
template <typename T, int E>
__device__ __forceinline__ void load_raw(const T* p, Raw<T, E>& r) {
  constexpr int kW = Raw<T, E>::kWords;
  static_assert(kW == 1 || kW == 2 || kW == 4, "4, 8 or 16 bytes");
  if constexpr (kW == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    r.w[0] = v.x, r.w[1] = v.y, r.w[2] = v.z, r.w[3] = v.w;
  } else if constexpr (kW == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    r.w[0] = v.x, r.w[1] = v.y;
  } else {
    r.w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}
template <typename T, int E>
__device__ __forceinline__ void raw_to_f(const Raw<T, E>& r, float (&f)[E]) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if constexpr (sizeof(T) == 2)
      f[e] = (e & 1) ? bf16_hi(r.w[e / 2]) : bf16_lo(r.w[e / 2]);
    else
      f[e] = __uint_as_float(r.w[e]);
  }
}

// Copies `bytes` (a multiple of 16, both addresses 16-byte aligned) with the
// 32 lanes of one warp.
__device__ __forceinline__ void block_copy_warp(void* dst, const void* src, int bytes, int lane) {
  uint4* d = reinterpret_cast<uint4*>(dst);
  const uint4* s = reinterpret_cast<const uint4*>(src);
  for (int i = lane; i < bytes / 16; i += 32) d[i] = s[i];
}

// ------------------------------------------------------------ tensor cores (mma.sync)

// Four 8 x 8 b16 matrices from shared memory: lane l gives the address of
// row (l mod 8) of matrix l / 8; register i holds matrix i in the mma
// fragment layout (lane 4g + t: row g, elements 2t and 2t + 1).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += A B for a 16 x 16 BF16 A (row-major fragment a) and a 16 x 8 BF16 B
// (column-major fragment b0, b1), FP32 accumulators: d[0..1] row g, d[2..3]
// row g + 8, columns 2t and 2t + 1 (lane 4g + t).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------ reductions

// Reduce-scatter across groups of L lanes: lane l holds L partial sums
// v[0..L-1]; on return lane l holds the total, over its group, of partial
// (l mod L). L - 1 shuffles instead of L * log2(L).
template <int L>
__device__ __forceinline__ float reduce_scatter(float (&v)[L], int lane) {
#pragma unroll
  for (int o = L / 2; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < o; ++k) {
      const float send = upper ? v[k] : v[k + o];
      const float keep = upper ? v[k + o] : v[k];
      v[k] = keep + __shfl_xor_sync(kFull, send, o);
    }
  }
  return v[0];
}

// ------------------------------------------------------------ row-dot engine
//
// A state tile sits in shared memory row-major, `COLS` elements of type TS
// per row. For 32 consecutive rows the engine computes dot(row, vec) with
// 16-byte loads: lane l reads chunk (l mod LPR) of row (k * RPI + l / LPR) at
// step k, so each group of 8 lanes reads 128 contiguous bytes (no bank
// conflicts), then a reduce-scatter leaves row
//   row0 + (l mod LPR) * RPI + l / LPR
// in lane l. Each lane needs only the vector elements of its own chunk.
template <int COLS, typename TS>
struct RowDot {
  static constexpr int kEpc = Chunk<TS>::kElems;        // elements per chunk
  static constexpr int kCpr = COLS / kEpc;              // chunks per row
  static constexpr int kLpr = kCpr < 32 ? kCpr : 32;    // lanes per row
  static constexpr int kRpi = 32 / kLpr;                // rows per step
  static_assert(kCpr == kLpr, "one chunk per lane per row");

  __device__ __forceinline__ static int chunk_of(int lane) { return lane % kLpr; }
  __device__ __forceinline__ static int row_of(int lane) {
    return (lane % kLpr) * kRpi + lane / kLpr;
  }

  // vec: this lane's kEpc vector elements (chunk chunk_of(lane)).
  __device__ __forceinline__ static float rows32(const TS* tile, int row0, const float (&vec)[kEpc],
                                                 int lane) {
    float acc[kLpr];
    const TS* base = tile + (size_t)(row0 + lane / kLpr) * COLS + chunk_of(lane) * kEpc;
#pragma unroll
    for (int k = 0; k < kLpr; ++k) {
      const uint4 raw = *reinterpret_cast<const uint4*>(base + (size_t)k * kRpi * COLS);
      float f[kEpc];
      unpack<TS>(raw, f);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < kEpc; ++e) s = fmaf(f[e], vec[e], s);
      acc[k] = s;
    }
    return reduce_scatter<kLpr>(acc, lane);
  }

  // Split form of rows32 for a consumer that frees the shared tile early:
  // load32 copies this lane's chunks of 32 rows into registers, dot32 does
  // the arithmetic and the reduce-scatter on them.
  __device__ __forceinline__ static void load32(const TS* tile, int row0, int lane,
                                                uint4 (&raw)[kLpr]) {
    const TS* base = tile + (size_t)(row0 + lane / kLpr) * COLS + chunk_of(lane) * kEpc;
#pragma unroll
    for (int k = 0; k < kLpr; ++k)
      raw[k] = *reinterpret_cast<const uint4*>(base + (size_t)k * kRpi * COLS);
  }
  __device__ __forceinline__ static float dot32(const uint4 (&raw)[kLpr], const float (&vec)[kEpc],
                                                int lane) {
    float acc[kLpr];
#pragma unroll
    for (int k = 0; k < kLpr; ++k) {
      float f[kEpc];
      unpack<TS>(raw[k], f);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < kEpc; ++e) s = fmaf(f[e], vec[e], s);
      acc[k] = s;
    }
    return reduce_scatter<kLpr>(acc, lane);
  }

  // Two independent 32-row groups at once (loads first, then both reductions).
  __device__ __forceinline__ static void rows32x2(const TS* tile, int row0a, int row0b,
                                                  const float (&vec)[kEpc], int lane, float& da,
                                                  float& db) {
    float acc_a[kLpr], acc_b[kLpr];
    const TS* ba = tile + (size_t)(row0a + lane / kLpr) * COLS + chunk_of(lane) * kEpc;
    const TS* bb = tile + (size_t)(row0b + lane / kLpr) * COLS + chunk_of(lane) * kEpc;
#pragma unroll
    for (int k = 0; k < kLpr; ++k) {
      const uint4 ra = *reinterpret_cast<const uint4*>(ba + (size_t)k * kRpi * COLS);
      const uint4 rb = *reinterpret_cast<const uint4*>(bb + (size_t)k * kRpi * COLS);
      float fa[kEpc], fb[kEpc];
      unpack<TS>(ra, fa);
      unpack<TS>(rb, fb);
      float sa = 0.f, sb = 0.f;
#pragma unroll
      for (int e = 0; e < kEpc; ++e) {
        sa = fmaf(fa[e], vec[e], sa);
        sb = fmaf(fb[e], vec[e], sb);
      }
      acc_a[k] = sa;
      acc_b[k] = sb;
    }
    da = reduce_scatter<kLpr>(acc_a, lane);
    db = reduce_scatter<kLpr>(acc_b, lane);
  }
};

// Marks the end of one block's share of a sequence's work; the block that
// completes the sequence (`units` of `total`) runs `last()` after every other
// block of that sequence has finished (and therefore read the pointers).
// Call from one thread.
template <typename F>
__device__ __forceinline__ void arrive_and_finish(int32_t* sync, int units, int total, F last) {
  __threadfence();
  const int old = atomicAdd(sync, units);
  if (old + units == total) {
    __threadfence();
    last();
    *sync = 0;
  }
}

// Tiles of one block (grid-stride over `tiles` tiles, H tiles per sequence)
// whose sequence folds: len + k_next > W, or force and len > 0 (with
// `flags`: the sequences whose flag is set instead). Sequences
// with out-of-range pointers get REPLAYSSM_SEQ_BAD_POINTER and are skipped. One parallel
// load of the pointers per block, so a launch with nothing to fold is cheap.
// The list order is arbitrary; every listed tile is independent.
constexpr int kMaxFoldTiles = 128;
struct FoldList {
  int count;
  int tile[kMaxFoldTiles];
  int len[kMaxFoldTiles];
  int head[kMaxFoldTiles];
};

// True when a sequence's ring pointers are in range (head < W, len <= W).
__device__ __forceinline__ bool pointers_ok(int head, int len, int W) {
  return head >= 0 && head < W && len >= 0 && len <= W;
}

__device__ __forceinline__ void collect_folds(FoldList& fl, long long tiles, int H,
                                              const int32_t* ring_len, const int32_t* ring_head,
                                              int32_t* status, int W, int k_next, int force,
                                              const int32_t* flags = nullptr) {
  if (threadIdx.x == 0) fl.count = 0;
  __syncthreads();
  for (int k = threadIdx.x; k < kMaxFoldTiles; k += blockDim.x) {
    const long long t = blockIdx.x + (long long)k * gridDim.x;
    if (t >= tiles) break;
    const int seq = (int)(t / H);
    const int len = ring_len[seq], head = ring_head[seq];
    if (!pointers_ok(head, len, W)) {
      if (t % H == 0) atomicOr(status + seq, REPLAYSSM_SEQ_BAD_POINTER);
    } else if (flags ? flags[seq] != 0 : (len + k_next > W || (force && len > 0))) {
      const int pos = atomicAdd(&fl.count, 1);
      fl.tile[pos] = (int)t;
      fl.len[pos] = len;
      fl.head[pos] = head;
    }
  }
  __syncthreads();
}

}  // namespace rs
