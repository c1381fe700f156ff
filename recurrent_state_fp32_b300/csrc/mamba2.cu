// Mamba-2 kernels: replay decode, consolidate (fold), conventional step.
//
// Layer type named on "NVIDIA présente ReplaySSM : accélérer le décodage des
// modèles hybrides Mamba et GDN", section "Pourquoi les hybrides sont devenus
// la norme"; the decode/consolidate split follows "NVIDIA y Princeton
// aceleran modelos híbridos al guardar entradas recientes en lugar del estado
// completo", paragraph 2. Per head the state h is P x N (N contiguous); with
// dA_i = exp(dt_i A_h) and the n buffered tokens after the checkpoint h_c
// (the newest being the current token):
//   y   = (prod_i dA_i) (h_c C) + sum_j w_j (C . B_j) x_j + D x,
//   w_j = dt_j prod_{i>j} dA_i = dt_j exp(A_h sum_{i>j} dt_i),
//   fold: h_c <- (prod_i dA_i) h_c + sum_j w_j x_j B_j^T.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace rs {
namespace {

struct M2Decode {
  int batch, H, G, P, W, hpb;  // hpb: heads per block
  const void* S;               // read copy (bf16) or checkpoint (f32)
  const float* A;
  const float* D;
  const void* x;
  const void* B;
  const void* C;
  const float* dt;
  float* y;
  void* ring_x;
  void* ring_B;
  void* ring_C;
  float* ring_dt;
  int32_t* head;
  int32_t* len;
  int32_t* status;
  int32_t* sync;
};

// Shared-memory carve-up of the decode block (byte offsets).
struct M2DecodeSmem {
  size_t tiles, bars, Cs, CB, coef, decay, extra, total;
  __host__ __device__ M2DecodeSmem(int hpb, int P, int N, int W, int ts_bytes) {
    tiles = 0;
    bars = (size_t)hpb * P * N * ts_bytes;
    Cs = bars + 8 * (size_t)hpb;
    CB = Cs + 4 * (size_t)hpb * N;
    coef = CB + 4 * (size_t)hpb * W;
    decay = coef + 4 * (size_t)hpb * W;
    extra = decay + 4 * (size_t)hpb;
    total = extra + 4 * (size_t)hpb * P;
  }
};

// One block: one sequence, heads [h0, h0 + nh). The block issues bulk copies
// of its nh state tiles first, appends the token to the ring and computes the
// buffer terms while the tiles are in flight, then streams the tiles through
// the row-dot engine. The block that finishes the sequence last bumps len.
template <int N, typename TS, typename TI>
__global__ void __launch_bounds__(kThreads) mamba2_decode_kernel(const M2Decode a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using RD = RowDot<N, TS>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, G = a.G, P = a.P, W = a.W;
  const int per_seq = (H + a.hpb - 1) / a.hpb;
  const int seq = blockIdx.x / per_seq;
  const int h0 = (blockIdx.x % per_seq) * a.hpb;
  const int nh = min(a.hpb, H - h0);
  const int len = a.len[seq];
  const int hd = a.head[seq];
  if (!pointers_ok(hd, len, W) || len + 1 > W) {
    if (h0 == 0 && tid == 0)
      atomicOr(a.status + seq, pointers_ok(hd, len, W) ? REPLAYSSM_SEQ_RING_FULL
                                                       : REPLAYSSM_SEQ_BAD_POINTER);
    return;
  }
  const int n = len + 1;

  const M2DecodeSmem L(a.hpb, P, N, W, sizeof(TS));
  TS* tiles = reinterpret_cast<TS*>(smem + L.tiles);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  float* Cs = reinterpret_cast<float*>(smem + L.Cs);
  float* CB = reinterpret_cast<float*>(smem + L.CB);
  float* coef = reinterpret_cast<float*>(smem + L.coef);
  float* decay = reinterpret_cast<float*>(smem + L.decay);
  float* extra = reinterpret_cast<float*>(smem + L.extra);
  const size_t tile_elems = (size_t)P * N;

  if (tid == 0) {
    for (int i = 0; i < nh; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint64_t pol = l2_evict_first_policy();
    const uint32_t bytes = (uint32_t)(tile_elems * sizeof(TS));
    const TS* src = reinterpret_cast<const TS*>(a.S) + ((size_t)seq * H + h0) * tile_elems;
    for (int i = 0; i < nh; ++i) {
      mbar_arrive_expect_tx(&bars[i], bytes);
      bulk_g2s(tiles + i * tile_elems, src + i * tile_elems, bytes, &bars[i], pol);
    }
  }

  // Append: the token goes to slot (head + len) mod W.
  const int slot = (hd + len) % W;
  const TI* xin = reinterpret_cast<const TI*>(a.x);
  const TI* Bin = reinterpret_cast<const TI*>(a.B);
  const TI* Cin = reinterpret_cast<const TI*>(a.C);
  const TI* rx = reinterpret_cast<const TI*>(a.ring_x);
  const TI* rB = reinterpret_cast<const TI*>(a.ring_B);
  block_copy16(reinterpret_cast<TI*>(a.ring_x) + (((size_t)seq * W + slot) * H + h0) * P,
               xin + ((size_t)seq * H + h0) * P, nh * P * (int)sizeof(TI));
  if (tid < nh)
    a.ring_dt[((size_t)seq * W + slot) * H + h0 + tid] = a.dt[(size_t)seq * H + h0 + tid];
  if (h0 == 0) {
    block_copy16(reinterpret_cast<TI*>(a.ring_B) + ((size_t)seq * W + slot) * G * N,
                 Bin + (size_t)seq * G * N, G * N * (int)sizeof(TI));
    if (a.ring_C)
      block_copy16(reinterpret_cast<TI*>(a.ring_C) + ((size_t)seq * W + slot) * G * N,
                   Cin + (size_t)seq * G * N, G * N * (int)sizeof(TI));
  }

  // C of each head (its group's C), as floats.
  const int hpg = H / G;
  for (int idx = tid; idx < nh * N; idx += kThreads) {
    const int i = idx / N, c = idx - i * N;
    Cs[idx] = to_f(Cin[((size_t)seq * G + (h0 + i) / hpg) * N + c]);
  }
  __syncthreads();

  // CB[i][j] = C . B_j for entries j < n (entry len is the current token).
  for (int pr = warp; pr < nh * n; pr += kWarps) {
    const int i = pr / n, j = pr - i * n;
    const int g = (h0 + i) / hpg;
    const TI* Bj = (j < len) ? rB + (((size_t)seq * W + (hd + j) % W) * G + g) * N
                             : Bin + ((size_t)seq * G + g) * N;
    float s = 0.f;
    for (int c = lane; c < N; c += 32) s = fmaf(Cs[i * N + c], to_f(Bj[c]), s);
    s = warp_sum(s);
    if (lane == 0) CB[i * W + j] = s;
  }
  __syncthreads();

  // Per-head weights, newest entry first: coef_j = w_j (C . B_j).
  if (tid < nh) {
    const int h = h0 + tid;
    const float Ah = a.A[h];
    float acc = 0.f;  // sum of dt over entries newer than j
    for (int j = n - 1; j >= 0; --j) {
      const float dtj = (j < len) ? a.ring_dt[((size_t)seq * W + (hd + j) % W) * H + h]
                                  : a.dt[(size_t)seq * H + h];
      coef[tid * W + j] = dtj * expf(Ah * acc) * CB[tid * W + j];
      acc += dtj;
    }
    decay[tid] = expf(Ah * acc);
  }
  __syncthreads();

  // extra[i][p] = sum_j coef_j x_j[p] + D x[p]
  for (int idx = tid; idx < nh * P; idx += kThreads) {
    const int i = idx / P, p = idx - i * P;
    const int h = h0 + i;
    const float xt = to_f(xin[((size_t)seq * H + h) * P + p]);
    float e = (a.D[h] + coef[i * W + len]) * xt;
#pragma unroll 4
    for (int j = 0; j < len; ++j)
      e = fmaf(coef[i * W + j], to_f(rx[(((size_t)seq * W + (hd + j) % W) * H + h) * P + p]), e);
    extra[idx] = e;
  }
  __syncthreads();

  // Stream the tiles: each pass is 32 rows of one head.
  const int passes = P / 32;
  bool ok = true;
  for (int ps = warp; ps < nh * passes; ps += kWarps) {
    const int i = ps / passes, row0 = (ps - i * passes) * 32;
    if (!mbar_wait(&bars[i], 0)) {
      ok = false;
      break;
    }
    float vec[RD::kEpc];
    const float* cv = Cs + i * N + RD::chunk_of(lane) * RD::kEpc;
#pragma unroll
    for (int e = 0; e < RD::kEpc; ++e) vec[e] = cv[e];
    const float dot = RD::rows32(tiles + i * tile_elems, row0, vec, lane);
    const int r = row0 + RD::row_of(lane);
    a.y[((size_t)seq * H + h0 + i) * P + r] = fmaf(decay[i], dot, extra[i * P + r]);
  }
  if (!ok) atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < nh; ++i) mbar_wait(&bars[i], 0);  // no copy may land after exit
    arrive_and_finish(a.sync + seq, nh, H, [&] { a.len[seq] = len + 1; });
  }
}

struct M2Fold {
  int batch, H, G, P, W, k_next, force;
  float* S;
  bf16* Sr;
  const float* A;
  const void* ring_x;
  const void* ring_B;
  const float* ring_dt;
  int32_t* head;
  int32_t* len;
  int32_t* status;
  int32_t* sync;
};

// Grid-stride over (sequence, head) tiles; only tiles of folding sequences do
// work. Per tile: stage B_j and w_j x_j in shared memory, then every float4 of
// the FP32 checkpoint is read once, updated in registers and written once
// (plus its bf16 read copy).
template <int N, typename TI>
__global__ void __launch_bounds__(kThreads) mamba2_fold_kernel(const M2Fold a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ FoldList fl;
  __shared__ float s_w[64];
  __shared__ float s_decay;
  const int tid = threadIdx.x;
  const int H = a.H, G = a.G, P = a.P, W = a.W;
  float* Bs = reinterpret_cast<float*>(smem);  // [W][N]
  float* xw = Bs + (size_t)W * N;              // [W][P]
  const TI* rx = reinterpret_cast<const TI*>(a.ring_x);
  const TI* rB = reinterpret_cast<const TI*>(a.ring_B);

  collect_folds(fl, (long long)a.batch * H, H, a.len, a.head, a.status, W, a.k_next, a.force);
  for (int f = 0; f < fl.count; ++f) {
    const int t = fl.tile[f], len = fl.len[f], hd = fl.head[f];
    const int seq = t / H, h = t - seq * H, g = h / (H / G);
    const int n = len;
    for (int idx = tid; idx < n * N; idx += kThreads) {
      const int j = idx / N, c = idx - j * N;
      Bs[idx] = to_f(rB[(((size_t)seq * W + (hd + j) % W) * G + g) * N + c]);
    }
    if (tid == 0) {
      const float Ah = a.A[h];
      float acc = 0.f;
      for (int j = n - 1; j >= 0; --j) {
        const float dtj = a.ring_dt[((size_t)seq * W + (hd + j) % W) * H + h];
        s_w[j] = dtj * expf(Ah * acc);
        acc += dtj;
      }
      s_decay = expf(Ah * acc);
    }
    __syncthreads();
    for (int idx = tid; idx < n * P; idx += kThreads) {
      const int j = idx / P, p = idx - j * P;
      xw[idx] = s_w[j] * to_f(rx[(((size_t)seq * W + (hd + j) % W) * H + h) * P + p]);
    }
    __syncthreads();
    const float decay = s_decay;
    float4* St = reinterpret_cast<float4*>(a.S + (size_t)t * P * N);
    uint2* Rt = a.Sr ? reinterpret_cast<uint2*>(a.Sr + (size_t)t * P * N) : nullptr;
    constexpr int kC4 = N / 4;  // float4 chunks per row
    const int chunks = P * kC4;
    constexpr int kU = 4;
    for (int base = tid; base < chunks; base += kThreads * kU) {
      float4 hv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int ci = base + u * kThreads;
        if (ci < chunks) hv[u] = St[ci];
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int ci = base + u * kThreads;
        if (ci >= chunks) break;
        const int p = ci / kC4, c4 = (ci - p * kC4) * 4;
        float r0 = decay * hv[u].x, r1 = decay * hv[u].y, r2 = decay * hv[u].z,
              r3 = decay * hv[u].w;
        for (int j = 0; j < n; ++j) {
          const float xv = xw[j * P + p];
          const float4 b = *reinterpret_cast<const float4*>(Bs + j * N + c4);
          r0 = fmaf(xv, b.x, r0);
          r1 = fmaf(xv, b.y, r1);
          r2 = fmaf(xv, b.z, r2);
          r3 = fmaf(xv, b.w, r3);
        }
        St[ci] = make_float4(r0, r1, r2, r3);
        if (Rt) Rt[ci] = make_uint2(pack_bf16x2(r0, r1), pack_bf16x2(r2, r3));
      }
    }
    __syncthreads();
    if (tid == 0)
      arrive_and_finish(a.sync + seq, 1, H, [&] {
        a.head[seq] = (hd + len) % W;
        a.len[seq] = 0;
      });
  }
}

struct M2Conv {
  int batch, H, G, P;
  float* S;
  const float* A;
  const float* D;
  const void* x;
  const void* B;
  const void* C;
  const float* dt;
  float* y;
};

// Conventional read-modify-write step: each warp owns 32 rows of one head,
// reads each float4 of h once, writes it back updated, and reduces h'.C with
// the same reduce-scatter as the replay kernels.
template <int N, typename TI>
__global__ void __launch_bounds__(kThreads) mamba2_conventional_kernel(const M2Conv a) {
  using RD = RowDot<N, float>;
  constexpr int kL = RD::kLpr, kR = RD::kRpi;
  const int lane = threadIdx.x & 31;
  const int passes = a.P / 32;
  const long long gw = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (gw >= (long long)a.batch * a.H * passes) return;
  const long long tile = gw / passes;
  const int row0 = (int)(gw - tile * passes) * 32;
  const int seq = (int)(tile / a.H), h = (int)(tile - (long long)seq * a.H);
  const int g = h / (a.H / a.G);
  const float dtv = a.dt[tile];
  const float dA = expf(dtv * a.A[h]);
  const TI* xin = reinterpret_cast<const TI*>(a.x) + tile * a.P;
  const int c0 = RD::chunk_of(lane) * 4;
  const TI* Bv = reinterpret_cast<const TI*>(a.B) + ((size_t)seq * a.G + g) * N + c0;
  const TI* Cv = reinterpret_cast<const TI*>(a.C) + ((size_t)seq * a.G + g) * N + c0;
  float bq[4], cq[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    bq[e] = to_f(Bv[e]);
    cq[e] = to_f(Cv[e]);
  }
  float4* base = reinterpret_cast<float4*>(a.S + tile * a.P * N + (size_t)(row0 + lane / kL) * N + c0);
  float acc[kL];
  constexpr int kHalf = kL > 16 ? kL / 2 : kL;
#pragma unroll
  for (int k0 = 0; k0 < kL; k0 += kHalf) {
    float4 hv[kHalf];
#pragma unroll
    for (int k = 0; k < kHalf; ++k) hv[k] = base[(size_t)(k0 + k) * kR * (N / 4)];
#pragma unroll
    for (int k = 0; k < kHalf; ++k) {
      const int row = row0 + (k0 + k) * kR + lane / kL;
      const float xr = dtv * to_f(xin[row]);
      float4 o;
      o.x = fmaf(xr, bq[0], dA * hv[k].x);
      o.y = fmaf(xr, bq[1], dA * hv[k].y);
      o.z = fmaf(xr, bq[2], dA * hv[k].z);
      o.w = fmaf(xr, bq[3], dA * hv[k].w);
      base[(size_t)(k0 + k) * kR * (N / 4)] = o;
      acc[k0 + k] = fmaf(o.x, cq[0], fmaf(o.y, cq[1], fmaf(o.z, cq[2], o.w * cq[3])));
    }
  }
  const float s = reduce_scatter<kL>(acc, lane);
  const int r = row0 + RD::row_of(lane);
  a.y[tile * a.P + r] = fmaf(a.D[h], to_f(xin[r]), s);
}

template <int N, typename TS, typename TI>
cudaError_t decode_inst(const M2Decode& a, cudaStream_t st) {
  const M2DecodeSmem L(a.hpb, a.P, N, a.W, sizeof(TS));
  auto kern = mamba2_decode_kernel<N, TS, TI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L.total);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)a.batch * ((a.H + a.hpb - 1) / a.hpb);
  kern<<<(unsigned)blocks, kThreads, L.total, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mamba2_decode(const replayssm_dims& d, const replayssm_state& s, const float* A,
                                 const float* D, const void* x, const void* B, const void* C,
                                 const float* dt, float* y, cudaStream_t st) {
  const bool rd16 = s.S_read != nullptr;
  const int ts = rd16 ? 2 : 4;
  const size_t tile_bytes = (size_t)d.dv * d.dk * ts;
  // About 64 KB of state per block (three blocks per SM); fewer heads per
  // block when the batch is too small to fill every SM twice.
  int hpb = (int)std::max<size_t>(1, (64 * 1024) / tile_bytes);
  hpb = std::min(hpb, d.heads);
  const int sms = device_info().sms;
  while (hpb > 1 && (long long)d.batch * ((d.heads + hpb - 1) / hpb) < 2LL * sms) hpb = (hpb + 1) / 2;
  M2Decode a{d.batch, d.heads, d.groups, d.dv, d.window, hpb,
             rd16 ? (const void*)s.S_read : (const void*)s.S_ckpt,
             A, D, x, B, C, dt, y, s.ring_x, s.ring_B, s.ring_C, s.ring_dt,
             s.ring_head, s.ring_len, s.status, s.sync};
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  if (d.dk == 128) {
    if (rd16) return in16 ? decode_inst<128, bf16, bf16>(a, st) : decode_inst<128, bf16, float>(a, st);
    return in16 ? decode_inst<128, float, bf16>(a, st) : decode_inst<128, float, float>(a, st);
  }
  if (rd16) return in16 ? decode_inst<64, bf16, bf16>(a, st) : decode_inst<64, bf16, float>(a, st);
  return in16 ? decode_inst<64, float, bf16>(a, st) : decode_inst<64, float, float>(a, st);
}

cudaError_t launch_mamba2_fold(const replayssm_dims& d, const replayssm_state& s, const float* A,
                               int k_next, int force, cudaStream_t st) {
  M2Fold a{d.batch, d.heads, d.groups, d.dv, d.window, k_next, force, s.S_ckpt,
           reinterpret_cast<bf16*>(s.S_read), A, s.ring_x, s.ring_B, s.ring_dt,
           s.ring_head, s.ring_len, s.status, s.sync};
  const long long tiles = (long long)d.batch * d.heads;
  const size_t smem = (size_t)d.window * (d.dk + d.dv) * sizeof(float);
  const int grid = fold_grid(tiles);
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  cudaError_t e;
  if (d.dk == 128) {
    auto kern = in16 ? mamba2_fold_kernel<128, bf16> : mamba2_fold_kernel<128, float>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(a);
  } else {
    auto kern = in16 ? mamba2_fold_kernel<64, bf16> : mamba2_fold_kernel<64, float>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_mamba2_conventional(const replayssm_dims& d, float* S, const float* A,
                                       const float* D, const void* x, const void* B, const void* C,
                                       const float* dt, float* y, cudaStream_t st) {
  M2Conv a{d.batch, d.heads, d.groups, d.dv, S, A, D, x, B, C, dt, y};
  const long long warps = (long long)d.batch * d.heads * (d.dv / 32);
  const unsigned grid = (unsigned)((warps + kWarps - 1) / kWarps);
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  if (d.dk == 128) {
    if (in16) mamba2_conventional_kernel<128, bf16><<<grid, kThreads, 0, st>>>(a);
    else mamba2_conventional_kernel<128, float><<<grid, kThreads, 0, st>>>(a);
  } else {
    if (in16) mamba2_conventional_kernel<64, bf16><<<grid, kThreads, 0, st>>>(a);
    else mamba2_conventional_kernel<64, float><<<grid, kThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace rs
