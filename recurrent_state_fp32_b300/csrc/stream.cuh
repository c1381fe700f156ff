// Streaming row-dot kernel shared by the replay decode paths.
//
// After a preparation kernel has reduced the ring to per-head values in the
// workspace (a vector v, a scale a and a per-row additive term e), every
// output row is
//     out[r] = a * (S[r, :] . v) + e[r]
// over the state rows S (the BF16 read copy or the FP32 checkpoint). This is
// the pure HBM stream of the method: each state byte is read once.
//
// Persistent blocks, one per SM. Work is split in units (sequence, head, row
// block of RB rows, about 16 KB of state): block b owns the units with flat
// index in [u0, u1). The last warp (producer) issues one bulk copy per unit
// into a ring of NS shared-memory stages (one large copy per unit: bulk
// copies have a fixed cost that small copies do not amortise). Consumer
// groups of GU warps take units round robin (group g: units g, g + NG, ...;
// stage i mod NS with NS a multiple of NG, so a stage always has the same
// group and mbarrier parity waits cannot alias); each warp of a group handles
// RB / GU rows. A consumer issues its unit's vector, scale and additive-term
// loads before it waits for the rows, copies its rows to registers when they
// fit and frees the stage at once, then reduces and writes the outputs.
#pragma once

#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace rs {

constexpr int kStreamGroups = 4;                              // consumer groups
constexpr int kStreamMaxThreads = 32 * (2 * kStreamGroups + 1);

struct StreamArgs {
  int batch, H, P, RB, nrb, NS, GU, K;
  const void* S;        // state rows [b, H, P, N]
  float* out;           // [b, K, H, P]
  const float* work;    // [b, K, H, wrow]
  int wrow;             // floats per work row
  int vec_off;          // vector offset in the work row; < 0: vector from vin
  int extra_off;        // additive-term offset in the work row
  int scale_off;        // scale offset in the work row; < 0: scale 1
  const int32_t* flags; // per sequence: nonzero = write outputs
  const void* vin;      // vector input [b, K, G, N] when vec_off < 0
  int G;                // groups of vin (head h uses group h / (H / G))
  int32_t* status;      // timeout reporting
};

__host__ __device__ inline size_t stream_stage_bytes(int RB, int N, int ts) {
  return align_up((size_t)RB * N * ts, 128);
}

// KMAX: compile-time bound on the vectors per unit (K <= KMAX), so that all
// per-vector registers are statically indexed.
template <int N, typename TS, typename TV, int KMAX>
__global__ void __launch_bounds__(kStreamMaxThreads, 1) stream_kernel(const StreamArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using RD = RowDot<N, TS>;
  constexpr int kE = RD::kEpc;
  // A warp's 32 rows fit in 64 registers per lane: copy out, free the stage early.
  constexpr bool kEarly = RD::kLpr <= 16;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CW = (int)(blockDim.x / 32) - 1;  // consumer warps; the producer is warp CW
  const int GU = a.GU, NG = CW / GU, NS = a.NS, H = a.H, P = a.P, RB = a.RB, nrb = a.nrb;
  const int K = a.K;
  const size_t stage = stream_stage_bytes(RB, N, sizeof(TS));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * stage);
  uint64_t* empty = full + NS;
  __shared__ int abort_smem;
  volatile int& abort_flag = abort_smem;
  const long long units = (long long)a.batch * H * nrb;
  const int u0 = (int)(units * blockIdx.x / gridDim.x);
  const int u1 = (int)(units * (blockIdx.x + 1) / gridDim.x);
  const uint32_t tile_bytes = (uint32_t)((size_t)RB * N * sizeof(TS));

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], GU);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();

  if (warp == CW) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_evict_first_policy();
    const TS* Sg = reinterpret_cast<const TS*>(a.S);
    int ps = 0;          // stage of the next unit
    uint32_t pk = 0;     // parity of the empty-barrier phase to wait for on stage ps
    bool pwrap = false;  // stages are being reused
    int hg = u0 / nrb, rb = u0 - (u0 / nrb) * nrb;  // global head, row block of unit u0
    for (int u = u0; u < u1; ++u) {
      const int s = ps;
      if (pwrap && !mbar_wait_warp(&empty[s], pk)) {
        if (lane == 0) abort_flag = 1;
        break;
      }
      if (++ps == NS) {
        ps = 0;
        if (pwrap) pk ^= 1;
        pwrap = true;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[s], tile_bytes);
        bulk_g2s(smem + (size_t)s * stage, Sg + ((size_t)hg * P + (size_t)rb * RB) * N, tile_bytes,
                 &full[s], pol);
      }
      if (++rb == nrb) {
        rb = 0;
        ++hg;
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int gi = warp / GU, part = warp - gi * GU;
    const int RBp = RB / GU;  // rows of a unit handled by this warp (a multiple of 32)
    auto group_any = [&](bool p) -> bool {
      if (GU == 1) return p;
      uint32_t res;
      asm volatile(
          "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
          " bar.red.or.pred po, %2, %3, pi;\n selp.u32 %0, 1, 0, po;\n}"
          : "=r"(res)
          : "r"((uint32_t)p), "r"(1 + gi), "r"(32 * GU)
          : "memory");
      return res != 0;
    };
    const int c0 = RD::chunk_of(lane) * kE;  // this lane's vector elements
    // The work rows come from the preparation grid (this grid may start
    // before it ends); the producer's state copies do not depend on it.
    griddep_wait();
    int s = gi;
    uint32_t ph = 0;
    for (int i = gi; u0 + i < u1; i += NG) {
      const int u = u0 + i;
      const int hg = u / nrb, rb = u - hg * nrb;
      const int seq = hg / H, h = hg - seq * H;
      const int row0 = rb * RB + part * RBp;  // first row of this warp within the head
      // Epilogue inputs first: their latency overlaps the wait for the rows.
      const bool write = a.flags[seq] != 0;
      const float* w0 = a.work + ((size_t)seq * K * H + h) * a.wrow;
      float vec[KMAX][kE];
      float scale[KMAX], extra[4];  // extra: single-vector case, per 32-row group
      const int ngr = RBp / 32;     // 32-row groups of this warp (1..4)
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k >= K) break;
        const float* wk = w0 + (size_t)k * H * a.wrow;
        if (a.vec_off >= 0) {
#pragma unroll
          for (int e = 0; e < kE; e += 4) {
            const float4 v4 = *reinterpret_cast<const float4*>(wk + a.vec_off + c0 + e);
            vec[k][e] = v4.x;
            vec[k][e + 1] = v4.y;
            vec[k][e + 2] = v4.z;
            vec[k][e + 3] = v4.w;
          }
        } else {
          const TV* vin = reinterpret_cast<const TV*>(a.vin) +
                          (((size_t)seq * K + k) * a.G + h / (H / a.G)) * N + c0;
#pragma unroll
          for (int e = 0; e < kE; ++e) vec[k][e] = to_f(vin[e]);
        }
        scale[k] = a.scale_off >= 0 ? wk[a.scale_off] : 1.f;
      }
      if constexpr (KMAX == 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < ngr) extra[q] = w0[a.extra_off + row0 + 32 * q + RD::row_of(lane)];
      }
      const bool aborted = __shfl_sync(kFull, abort_flag, 0) != 0;
      const bool landed = !aborted && mbar_wait_warp(&full[s], ph);
      if (!aborted && !landed && lane == 0) {
        abort_flag = 1;
        atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
      }
      if (group_any(!landed)) break;  // one decision per group
      const TS* tile = reinterpret_cast<const TS*>(smem + (size_t)s * stage) + (size_t)part * RBp * N;
      float* yrow = a.out + ((size_t)seq * K * H + h) * P + row0;
      if constexpr (KMAX > 1) {
        // Several vectors: read the tile from shared memory once per chunk of
        // KC vectors (KC * kLpr accumulators stay in registers); the additive
        // terms are loaded per 32-row group.
        constexpr int KC = KMAX < 64 / RD::kLpr ? KMAX : 64 / RD::kLpr;
#pragma unroll 1
        for (int q = 0; q < ngr; ++q) {
          const int r = 32 * q + RD::row_of(lane);
#pragma unroll 1
          for (int k0 = 0; k0 < KMAX; k0 += KC) {
            if (k0 >= K) break;
            float ex[KC];
#pragma unroll
            for (int c = 0; c < KC; ++c)
              ex[c] = k0 + c < K ? w0[(size_t)(k0 + c) * H * a.wrow + a.extra_off + row0 + r] : 0.f;
            float acc[KC][RD::kLpr];
            const TS* base = tile + (size_t)(32 * q + lane / RD::kLpr) * N + c0;
#pragma unroll
            for (int kk = 0; kk < RD::kLpr; ++kk) {
              const uint4 raw = *reinterpret_cast<const uint4*>(base + (size_t)kk * RD::kRpi * N);
              float f[kE];
              unpack<TS>(raw, f);
#pragma unroll
              for (int c = 0; c < KC; ++c) {
                float sacc = 0.f;
#pragma unroll
                for (int e = 0; e < kE; ++e) sacc = fmaf(f[e], vec[k0 + c][e], sacc);
                acc[c][kk] = sacc;
              }
            }
#pragma unroll
            for (int c = 0; c < KC; ++c) {
              if (k0 + c >= K) break;
              const float d = reduce_scatter<RD::kLpr>(acc[c], lane);
              if (write) yrow[(size_t)(k0 + c) * H * P + r] = fmaf(scale[k0 + c], d, ex[c]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      } else if (kEarly && ngr == 1) {
        uint4 raw[RD::kLpr];
        RD::load32(tile, 0, lane, raw);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        const float d = RD::dot32(raw, vec[0], lane);
        if (write) yrow[RD::row_of(lane)] = fmaf(scale[0], d, extra[0]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q >= ngr) break;
          const float d = RD::rows32(tile, 32 * q, vec[0], lane);
          if (write) yrow[32 * q + RD::row_of(lane)] = fmaf(scale[0], d, extra[q]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      s += NG;
      if (s >= NS) {
        s -= NS;
        ph ^= 1;
      }
    }
  }
  __syncthreads();
  // No bulk copy may land after the block exits.
  if (tid == 0 && abort_flag) {
    for (int s = 0; s < NS; ++s) {
      mbar_wait(&full[s], 0);
      mbar_wait(&full[s], 1);
    }
  }
}

// Tile shape, consumer layout and stage count for a stream over heads of P
// rows by N columns of TS; launches stream_kernel<N, TS, TV>.
template <int N, typename TS, typename TV, int KMAX>
cudaError_t launch_stream(StreamArgs a, cudaStream_t st) {
  const DeviceInfo& dev = device_info();
  // About 16 KB of state rows per unit (at least 32 rows, dividing P).
  int RB = std::max(32, (int)(16384 / (N * sizeof(TS))) / 32 * 32);
  RB = std::min(RB, a.P);
  while (a.P % RB) RB -= 32;
  a.RB = RB;
  a.nrb = a.P / RB;
  a.GU = RB % 64 == 0 ? 2 : 1;  // each warp's share must be whole 32-row groups
  if (RB / a.GU > 128 || a.K > KMAX) return cudaErrorInvalidValue;
  const size_t stage = stream_stage_bytes(RB, N, sizeof(TS));
  const int fit = (int)(((size_t)dev.smem_optin - 2048) / (stage + 16));
  const int NS = std::min(fit, 3 * kStreamGroups) / kStreamGroups * kStreamGroups;
  if (NS < kStreamGroups) return cudaErrorInvalidConfiguration;
  a.NS = NS;
  const size_t smem = (size_t)NS * stage + 2 * (size_t)NS * 8;
  auto kern = stream_kernel<N, TS, TV, KMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.batch * a.H * a.nrb;
  if (units >= (1LL << 31)) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>(units, dev.sms);
  // Launched as a programmatic dependent of the preparation kernel before it
  // on the stream: blocks start (and stream state rows) as SMs free up.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(32 * (kStreamGroups * a.GU + 1));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace rs
