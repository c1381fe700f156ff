// Gated DeltaNet / KDA kernels: replay decode, speculative verify,
// consolidate (fold), conventional step.
//
// Layer types named on "NVIDIA présente ReplaySSM : accélérer le décodage des
// modèles hybrides Mamba et GDN", section "Pourquoi les hybrides sont devenus
// la norme". A head's state S is d_v x d_k (d_k contiguous) and
//   S_t = S_{t-1} A_t + beta_t v_t k_t^T,  A_t = Diag(alpha_t)(I - beta_t k_t k_t^T),
//   o_t = scale * S_t q_t,
// with a scalar gate (GDN) or a per-key-channel gate (KDA). Replay from the
// checkpoint S_c over the n buffered entries (newest = current token), as on
// "NVIDIA y Princeton aceleran modelos híbridos…", paragraph 2:
//   u <- scale q; for j = n..1: s = k_j.u; o += beta_j s v_j; u <- A_j u;
//   o += S_c u.
// Verify (same page, paragraph 3) runs that sweep once per draft and reads
// S_c once for all drafts. The fold applies the n updates row by row in FP32
// registers: s <- alpha (.) s; s <- s + beta (v_r - s.k) k.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace rs {
namespace {

struct DDecode {
  int batch, H, DV, W, nrb, K;  // nrb: row blocks per head; K: drafts (verify)
  const void* S;
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  float scale;
  float* o;
  void* ring_q;
  void* ring_k;
  void* ring_v;
  float* ring_alpha;
  float* ring_beta;
  int32_t* head;
  int32_t* len;
  int32_t* status;
  int32_t* sync;
};

// Shared-memory carve-up for decode (K = 1) and verify (K drafts).
struct DSmem {
  size_t tile, bar, kbuf, abuf, bbuf, vbuf, ubuf, coef, obuf, total;
  __host__ __device__ DSmem(int RB, int DK, int W, int K, bool kda, int ts_bytes) {
    tile = 0;
    bar = (size_t)RB * DK * ts_bytes;
    kbuf = bar + 16;
    abuf = kbuf + 4 * (size_t)W * DK;
    bbuf = abuf + 4 * (size_t)W * (kda ? DK : 1);
    vbuf = bbuf + 4 * (size_t)W;
    ubuf = vbuf + 4 * (size_t)W * RB;
    coef = ubuf + 4 * (size_t)K * DK;
    obuf = coef + 4 * (size_t)K * W;
    total = obuf + 4 * (size_t)K * RB;
  }
};

// Entry j of a sequence: j < len is ring slot (head + j) mod W; later entries
// come from the call's own inputs (the current token or draft j - len).
template <int DK, typename TI, bool KDA>
__device__ __forceinline__ void stage_entries(const DDecode& a, int seq, int h, int rb, int RB,
                                              int len, int hd, int n, float* kbuf, float* abuf,
                                              float* bbuf, float* vbuf) {
  const int H = a.H, W = a.W, DV = a.DV;
  const TI* rk = reinterpret_cast<const TI*>(a.ring_k);
  const TI* rv = reinterpret_cast<const TI*>(a.ring_v);
  const TI* ik = reinterpret_cast<const TI*>(a.k);
  const TI* iv = reinterpret_cast<const TI*>(a.v);
  // ring rows of (seq, h): vector fields [b, H, W, d], scalar fields [b, H, Wd];
  // inputs [b, K, H, ...]
  const int Wd = ring_wd(W);
  auto ring_ix = [&](int j) { return ((size_t)seq * H + h) * W + (hd + j) % W; };
  auto ring_sx = [&](int j) { return ((size_t)seq * H + h) * Wd + (hd + j) % W; };
  auto in_ix = [&](int j) { return ((size_t)seq * a.K + (j - len)) * H + h; };
  for (int idx = threadIdx.x; idx < n * DK; idx += kThreads) {
    const int j = idx / DK, c = idx - j * DK;
    kbuf[idx] = to_f(j < len ? rk[ring_ix(j) * DK + c] : ik[in_ix(j) * DK + c]);
    if (KDA) abuf[idx] = j < len ? a.ring_alpha[ring_ix(j) * DK + c] : a.alpha[in_ix(j) * DK + c];
  }
  for (int idx = threadIdx.x; idx < n * RB; idx += kThreads) {
    const int j = idx / RB, r = idx - j * RB + rb * RB;
    vbuf[idx] = to_f(j < len ? rv[ring_ix(j) * DV + r] : iv[in_ix(j) * DV + r]);
  }
  for (int j = threadIdx.x; j < n; j += kThreads) {
    bbuf[j] = j < len ? a.ring_beta[ring_sx(j)] : a.beta[in_ix(j)];
    if (!KDA) abuf[j] = j < len ? a.ring_alpha[ring_sx(j)] : a.alpha[in_ix(j)];
  }
}

// Writes input entry i (token or draft) of (seq, h) into ring slot `slot`.
template <int DK, typename TI, bool KDA>
__device__ __forceinline__ void append_entry(const DDecode& a, int seq, int h, int i, int slot) {
  const int H = a.H, W = a.W, DV = a.DV;
  const size_t in_ix = ((size_t)seq * a.K + i) * H + h;
  const size_t ring_ix = ((size_t)seq * H + h) * W + slot;
  const size_t ring_sx = ((size_t)seq * H + h) * ring_wd(W) + slot;
  block_copy16(reinterpret_cast<TI*>(a.ring_k) + ring_ix * DK,
               reinterpret_cast<const TI*>(a.k) + in_ix * DK, DK * (int)sizeof(TI));
  block_copy16(reinterpret_cast<TI*>(a.ring_v) + ring_ix * DV,
               reinterpret_cast<const TI*>(a.v) + in_ix * DV, DV * (int)sizeof(TI));
  if (a.ring_q)
    block_copy16(reinterpret_cast<TI*>(a.ring_q) + ring_ix * DK,
                 reinterpret_cast<const TI*>(a.q) + in_ix * DK, DK * (int)sizeof(TI));
  if (KDA) block_copy16(a.ring_alpha + ring_ix * DK, a.alpha + in_ix * DK, DK * 4);
  if (threadIdx.x == 0) {
    a.ring_beta[ring_sx] = a.beta[in_ix];
    if (!KDA) a.ring_alpha[ring_sx] = a.alpha[in_ix];
  }
}

// Backward sweep for one query by one warp over entries last..0; leaves u in
// ubuf and beta_j (k_j . u) in coef[j]. Lane l owns u[l*EPL .. l*EPL+EPL).
template <int DK, bool KDA>
__device__ __forceinline__ void sweep(const float* qv, int last, const float* kbuf,
                                      const float* abuf, const float* bbuf, float* ubuf,
                                      float* coef, int lane) {
  constexpr int EPL = DK / 32;
  float u[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) u[e] = qv[lane * EPL + e];
  for (int j = last; j >= 0; --j) {
    const float* kj = kbuf + j * DK + lane * EPL;
    float kk[EPL];
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kk[e] = kj[e];
      s = fmaf(kk[e], u[e], s);
    }
    s = warp_sum(s);
    const float bs = bbuf[j] * s;
    if (lane == 0) coef[j] = bs;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float g = KDA ? abuf[j * DK + lane * EPL + e] : abuf[j];
      u[e] = (u[e] - bs * kk[e]) * g;
    }
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) ubuf[lane * EPL + e] = u[e];
}

// One block per (sequence, head, row block). K == 1 is the decode step
// (appends and commits the token); K > 1 is the speculative verify (appends
// K drafts, commits nothing, one output per draft).
template <int DK, typename TS, typename TI, bool KDA, bool VERIFY>
__global__ void __launch_bounds__(kThreads) delta_replay_kernel(const DDecode a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using RD = RowDot<DK, TS>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, DV = a.DV, W = a.W, K = a.K;
  const int RB = DV / a.nrb;
  const int per_seq = H * a.nrb;
  const int seq = blockIdx.x / per_seq;
  const int rem = blockIdx.x - seq * per_seq;
  const int h = rem / a.nrb, rb = rem - h * a.nrb;
  const int len = a.len[seq];
  const int hd = a.head[seq];
  if (!pointers_ok(hd, len, W) || len + K > W) {
    if (rem == 0 && tid == 0)
      atomicOr(a.status + seq, pointers_ok(hd, len, W) ? REPLAYSSM_SEQ_RING_FULL
                                                       : REPLAYSSM_SEQ_BAD_POINTER);
    return;
  }
  const DSmem L(RB, DK, W, K, KDA, sizeof(TS));
  TS* tile = reinterpret_cast<TS*>(smem + L.tile);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
  float* kbuf = reinterpret_cast<float*>(smem + L.kbuf);
  float* abuf = reinterpret_cast<float*>(smem + L.abuf);
  float* bbuf = reinterpret_cast<float*>(smem + L.bbuf);
  float* vbuf = reinterpret_cast<float*>(smem + L.vbuf);
  float* ubuf = reinterpret_cast<float*>(smem + L.ubuf);
  float* coef = reinterpret_cast<float*>(smem + L.coef);
  float* obuf = reinterpret_cast<float*>(smem + L.obuf);

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)((size_t)RB * DK * sizeof(TS));
    const TS* src = reinterpret_cast<const TS*>(a.S) + (((size_t)seq * H + h) * DV + (size_t)rb * RB) * DK;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(tile, src, bytes, bar, l2_evict_first_policy());
  }
  if (rb == 0)
    for (int i = 0; i < K; ++i) append_entry<DK, TI, KDA>(a, seq, h, i, (hd + len + i) % W);
  const int n = len + K;
  stage_entries<DK, TI, KDA>(a, seq, h, rb, RB, len, hd, n, kbuf, abuf, bbuf, vbuf);
  __syncthreads();

  // One backward sweep per query (warp i handles drafts i, i+4, ...).
  const TI* qin = reinterpret_cast<const TI*>(a.q);
  for (int i = warp; i < K; i += kWarps) {
    float* qs = ubuf + i * DK;  // staged scaled query, overwritten by u
    for (int c = lane; c < DK; c += 32)
      qs[c] = a.scale * to_f(qin[(((size_t)seq * K + i) * H + h) * DK + c]);
    __syncwarp();
    sweep<DK, KDA>(qs, len + i, kbuf, abuf, bbuf, qs, coef + i * W, lane);
  }
  __syncthreads();
  // Buffer terms: obuf[i][r] = sum_{j <= len+i} beta_j s_j v_j[r].
  for (int idx = tid; idx < K * RB; idx += kThreads) {
    const int i = idx / RB, r = idx - i * RB;
    float s = 0.f;
    for (int j = 0; j <= len + i; ++j) s = fmaf(coef[i * W + j], vbuf[j * RB + r], s);
    obuf[idx] = s;
  }
  __syncthreads();

  // S_c u for every query from the one staged tile.
  const int passes = RB / 32;
  bool ok = true;
  for (int task = warp; task < K * passes; task += kWarps) {
    const int i = task / passes, row0 = (task - i * passes) * 32;
    if (!mbar_wait(bar, 0)) {
      ok = false;
      break;
    }
    float vec[RD::kEpc];
    const float* uv = ubuf + i * DK + RD::chunk_of(lane) * RD::kEpc;
#pragma unroll
    for (int e = 0; e < RD::kEpc; ++e) vec[e] = uv[e];
    const float dot = RD::rows32(tile, row0, vec, lane);
    const int r = row0 + RD::row_of(lane);
    a.o[(((size_t)seq * K + i) * H + h) * DV + (size_t)rb * RB + r] = dot + obuf[i * RB + r];
  }
  if (!ok) atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
  __syncthreads();
  if (tid == 0) {
    mbar_wait(bar, 0);  // no copy may land after exit
    if (!VERIFY) arrive_and_finish(a.sync + seq, 1, per_seq, [&] { a.len[seq] = len + 1; });
  }
}

struct DFold {
  int batch, H, DV, W, k_next, force;
  float* S;
  bf16* Sr;
  const void* ring_k;
  const void* ring_v;
  const float* ring_alpha;
  const float* ring_beta;
  int32_t* head;
  int32_t* len;
  int32_t* status;
  int32_t* sync;
};

// Grid-stride over (sequence, head) tiles of folding sequences. Rows are
// independent: 4 lanes per row, 8 rows per warp step; lane q of a row owns
// the float4 chunks q, q+4, q+8, ... (so 4 lanes read 64 contiguous bytes).
template <int DK, typename TI, bool KDA>
__global__ void __launch_bounds__(kThreads) delta_fold_kernel(const DFold a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ FoldList fl;
  constexpr int CH = DK / 16;  // float4 chunks per lane
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, DV = a.DV, W = a.W;
  float* kbuf = reinterpret_cast<float*>(smem);                  // [W][DK]
  float* abuf = kbuf + (size_t)W * DK;                           // [W][DK] or [W]
  float* bbuf = abuf + (size_t)W * (KDA ? DK : 1);               // [W]
  float* vbuf = bbuf + W;                                        // [W][DV]
  const TI* rk = reinterpret_cast<const TI*>(a.ring_k);
  const TI* rv = reinterpret_cast<const TI*>(a.ring_v);

  collect_folds(fl, (long long)a.batch * H, H, a.len, a.head, a.status, W, a.k_next, a.force);
  for (int f = 0; f < fl.count; ++f) {
    const int t = fl.tile[f], len = fl.len[f], hd = fl.head[f];
    const int seq = t / H, h = t - seq * H;
    const int n = len;
    auto ring_ix = [&](int j) { return ((size_t)seq * H + h) * W + (hd + j) % W; };
    auto ring_sx = [&](int j) { return ((size_t)seq * H + h) * ring_wd(W) + (hd + j) % W; };
    for (int idx = tid; idx < n * DK; idx += kThreads) {
      const int j = idx / DK, c = idx - j * DK;
      kbuf[idx] = to_f(rk[ring_ix(j) * DK + c]);
      if (KDA) abuf[idx] = a.ring_alpha[ring_ix(j) * DK + c];
    }
    for (int idx = tid; idx < n * DV; idx += kThreads) {
      const int j = idx / DV, r = idx - j * DV;
      vbuf[idx] = to_f(rv[ring_ix(j) * DV + r]);
    }
    for (int j = tid; j < n; j += kThreads) {
      bbuf[j] = a.ring_beta[ring_sx(j)];
      if (!KDA) abuf[j] = a.ring_alpha[ring_sx(j)];
    }
    __syncthreads();
    const int q = lane & 3;
    for (int r = warp * 8 + (lane >> 2); r < DV; r += kWarps * 8) {
      float4* row = reinterpret_cast<float4*>(a.S + ((size_t)t * DV + r) * DK);
      float s[CH][4];
#pragma unroll
      for (int m = 0; m < CH; ++m) {
        const float4 v4 = row[q + 4 * m];
        s[m][0] = v4.x;
        s[m][1] = v4.y;
        s[m][2] = v4.z;
        s[m][3] = v4.w;
      }
      for (int j = 0; j < n; ++j) {
        const float* kj = kbuf + j * DK;
        float d = 0.f;
#pragma unroll
        for (int m = 0; m < CH; ++m) {
          const float4 k4 = *reinterpret_cast<const float4*>(kj + (q + 4 * m) * 4);
          if (KDA) {
            const float4 a4 = *reinterpret_cast<const float4*>(abuf + j * DK + (q + 4 * m) * 4);
            s[m][0] *= a4.x;
            s[m][1] *= a4.y;
            s[m][2] *= a4.z;
            s[m][3] *= a4.w;
          } else {
            const float g = abuf[j];
#pragma unroll
            for (int e = 0; e < 4; ++e) s[m][e] *= g;
          }
          d = fmaf(s[m][0], k4.x, d);
          d = fmaf(s[m][1], k4.y, d);
          d = fmaf(s[m][2], k4.z, d);
          d = fmaf(s[m][3], k4.w, d);
        }
        d += __shfl_xor_sync(kFull, d, 1);
        d += __shfl_xor_sync(kFull, d, 2);
        const float c = bbuf[j] * (vbuf[j * DV + r] - d);
#pragma unroll
        for (int m = 0; m < CH; ++m) {
          const float4 k4 = *reinterpret_cast<const float4*>(kj + (q + 4 * m) * 4);
          s[m][0] = fmaf(c, k4.x, s[m][0]);
          s[m][1] = fmaf(c, k4.y, s[m][1]);
          s[m][2] = fmaf(c, k4.z, s[m][2]);
          s[m][3] = fmaf(c, k4.w, s[m][3]);
        }
      }
#pragma unroll
      for (int m = 0; m < CH; ++m) row[q + 4 * m] = make_float4(s[m][0], s[m][1], s[m][2], s[m][3]);
      if (a.Sr) {
        uint2* rrow = reinterpret_cast<uint2*>(a.Sr + ((size_t)t * DV + r) * DK);
#pragma unroll
        for (int m = 0; m < CH; ++m)
          rrow[q + 4 * m] = make_uint2(pack_bf16x2(s[m][0], s[m][1]), pack_bf16x2(s[m][2], s[m][3]));
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

struct DConv {
  int batch, H, DV;
  float* S;
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  float scale;
  float* o;
};

// Conventional read-modify-write step: one warp per 8 rows of one head, 8
// lanes per row (lane l of a row owns float4 chunks l, l+8, ...). Both dots
// of a row, (S Diag(alpha)) k and (S Diag(alpha)) q, come from one pass; the
// updated row is written back and o_r = scale (g.q + c (k.q)).
template <int DK, typename TI, bool KDA>
__global__ void __launch_bounds__(kThreads) delta_conventional_kernel(const DConv a) {
  constexpr int CH = DK / 32;  // float4 chunks per lane
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int groups = a.DV / 8;
  if (gw >= (long long)a.batch * a.H * groups) return;
  const long long t = gw / groups;
  const int r0 = (int)(gw - t * groups) * 8;
  const int sub = lane >> 3, c8 = lane & 7;
  const TI* qi = reinterpret_cast<const TI*>(a.q) + t * DK;
  const TI* ki = reinterpret_cast<const TI*>(a.k) + t * DK;
  const TI* vi = reinterpret_cast<const TI*>(a.v) + t * a.DV;
  float kq[CH][4], qq[CH][4], al[CH][4];
  float kqdot = 0.f;
#pragma unroll
  for (int m = 0; m < CH; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = (c8 + 8 * m) * 4 + e;
      kq[m][e] = to_f(ki[c]);
      qq[m][e] = to_f(qi[c]);
      al[m][e] = KDA ? a.alpha[t * DK + c] : a.alpha[t];
      kqdot = fmaf(kq[m][e], qq[m][e], kqdot);
    }
  kqdot += __shfl_xor_sync(kFull, kqdot, 1);
  kqdot += __shfl_xor_sync(kFull, kqdot, 2);
  kqdot += __shfl_xor_sync(kFull, kqdot, 4);
  const float be = a.beta[t];
  float4 sv[2][CH];
#pragma unroll
  for (int st = 0; st < 2; ++st) {
    const float4* row = reinterpret_cast<const float4*>(a.S + (t * a.DV + r0 + st * 4 + sub) * DK);
#pragma unroll
    for (int m = 0; m < CH; ++m) sv[st][m] = row[c8 + 8 * m];
  }
#pragma unroll
  for (int st = 0; st < 2; ++st) {
    const int r = r0 + st * 4 + sub;
    float g[CH][4];
    float d1 = 0.f, d2 = 0.f;
#pragma unroll
    for (int m = 0; m < CH; ++m) {
      g[m][0] = sv[st][m].x * al[m][0];
      g[m][1] = sv[st][m].y * al[m][1];
      g[m][2] = sv[st][m].z * al[m][2];
      g[m][3] = sv[st][m].w * al[m][3];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        d1 = fmaf(g[m][e], kq[m][e], d1);
        d2 = fmaf(g[m][e], qq[m][e], d2);
      }
    }
#pragma unroll
    for (int o = 1; o <= 4; o <<= 1) {
      d1 += __shfl_xor_sync(kFull, d1, o);
      d2 += __shfl_xor_sync(kFull, d2, o);
    }
    const float c = be * (to_f(vi[r]) - d1);
    float4* row = reinterpret_cast<float4*>(a.S + (t * a.DV + r) * DK);
#pragma unroll
    for (int m = 0; m < CH; ++m)
      row[c8 + 8 * m] = make_float4(fmaf(c, kq[m][0], g[m][0]), fmaf(c, kq[m][1], g[m][1]),
                                    fmaf(c, kq[m][2], g[m][2]), fmaf(c, kq[m][3], g[m][3]));
    if (c8 == 0) a.o[t * a.DV + r] = a.scale * fmaf(c, kqdot, d2);
  }
}

template <int DK, typename TS, typename TI, bool KDA, bool VERIFY>
cudaError_t replay_inst(const DDecode& a, cudaStream_t st) {
  const int RB = a.DV / a.nrb;
  const DSmem L(RB, DK, a.W, a.K, KDA, sizeof(TS));
  auto kern = delta_replay_kernel<DK, TS, TI, KDA, VERIFY>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)a.batch * a.H * a.nrb;
  kern<<<(unsigned)blocks, kThreads, L.total, st>>>(a);
  return cudaGetLastError();
}

template <bool VERIFY>
cudaError_t replay_dispatch(const replayssm_dims& d, const DDecode& a, bool rd16, cudaStream_t st) {
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  const bool kda = d.kind == REPLAYSSM_KDA;
#define RS_REPLAY(DK_)                                                                          \
  if (rd16) {                                                                                   \
    if (in16) return kda ? replay_inst<DK_, bf16, bf16, true, VERIFY>(a, st)                    \
                         : replay_inst<DK_, bf16, bf16, false, VERIFY>(a, st);                  \
    return kda ? replay_inst<DK_, bf16, float, true, VERIFY>(a, st)                             \
               : replay_inst<DK_, bf16, float, false, VERIFY>(a, st);                           \
  }                                                                                             \
  if (in16) return kda ? replay_inst<DK_, float, bf16, true, VERIFY>(a, st)                     \
                       : replay_inst<DK_, float, bf16, false, VERIFY>(a, st);                   \
  return kda ? replay_inst<DK_, float, float, true, VERIFY>(a, st)                              \
             : replay_inst<DK_, float, float, false, VERIFY>(a, st);
  if (d.dk == 128) {
    RS_REPLAY(128)
  }
  RS_REPLAY(64)
#undef RS_REPLAY
}

// Row blocks per head: split heads when the batch cannot fill the SMs.
int pick_row_blocks(const replayssm_dims& d) {
  int nrb = 1;
  const int sms = device_info().sms;
  while (nrb < 8 && d.dv / (nrb * 2) >= 32 && (d.dv / (nrb * 2)) % 32 == 0 &&
         (long long)d.batch * d.heads * nrb < 2LL * sms)
    nrb *= 2;
  return nrb;
}

DDecode make_args(const replayssm_dims& d, const replayssm_state& s, int K, const void* q,
                  const void* k, const void* v, const float* alpha, const float* beta,
                  float scale, float* o) {
  return DDecode{d.batch, d.heads, d.dv, d.window, pick_row_blocks(d), K,
                 s.S_read ? (const void*)s.S_read : (const void*)s.S_ckpt,
                 q, k, v, alpha, beta, scale, o,
                 s.ring_q, s.ring_k, s.ring_v, s.ring_alpha, s.ring_beta,
                 s.ring_head, s.ring_len, s.status, s.sync};
}

}  // namespace

cudaError_t launch_delta_decode(const replayssm_dims& d, const replayssm_state& s, const void* q,
                                const void* k, const void* v, const float* alpha,
                                const float* beta, float scale, float* o, cudaStream_t st) {
  return replay_dispatch<false>(d, make_args(d, s, 1, q, k, v, alpha, beta, scale, o),
                                s.S_read != nullptr, st);
}

cudaError_t launch_delta_verify(const replayssm_dims& d, const replayssm_state& s, int K,
                                const void* q, const void* k, const void* v, const float* alpha,
                                const float* beta, float scale, float* o, cudaStream_t st) {
  return replay_dispatch<true>(d, make_args(d, s, K, q, k, v, alpha, beta, scale, o),
                               s.S_read != nullptr, st);
}

cudaError_t launch_delta_fold(const replayssm_dims& d, const replayssm_state& s, int k_next,
                              int force, cudaStream_t st) {
  DFold a{d.batch, d.heads, d.dv, d.window, k_next, force, s.S_ckpt,
          reinterpret_cast<bf16*>(s.S_read), s.ring_k, s.ring_v, s.ring_alpha, s.ring_beta,
          s.ring_head, s.ring_len, s.status, s.sync};
  const bool kda = d.kind == REPLAYSSM_KDA;
  const size_t smem =
      4 * ((size_t)d.window * d.dk + (size_t)d.window * (kda ? d.dk : 1) + d.window +
           (size_t)d.window * d.dv);
  const int grid = fold_grid((long long)d.batch * d.heads);
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  void (*kern)(const DFold);
  if (d.dk == 128)
    kern = in16 ? (kda ? delta_fold_kernel<128, bf16, true> : delta_fold_kernel<128, bf16, false>)
                : (kda ? delta_fold_kernel<128, float, true> : delta_fold_kernel<128, float, false>);
  else
    kern = in16 ? (kda ? delta_fold_kernel<64, bf16, true> : delta_fold_kernel<64, bf16, false>)
                : (kda ? delta_fold_kernel<64, float, true> : delta_fold_kernel<64, float, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_delta_conventional(const replayssm_dims& d, float* S, const void* q,
                                      const void* k, const void* v, const float* alpha,
                                      const float* beta, float scale, float* o, cudaStream_t st) {
  DConv a{d.batch, d.heads, d.dv, S, q, k, v, alpha, beta, scale, o};
  const long long warps = (long long)d.batch * d.heads * (d.dv / 8);
  const unsigned grid = (unsigned)((warps + kWarps - 1) / kWarps);
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  const bool kda = d.kind == REPLAYSSM_KDA;
  void (*kern)(const DConv);
  if (d.dk == 128)
    kern = in16 ? (kda ? delta_conventional_kernel<128, bf16, true> : delta_conventional_kernel<128, bf16, false>)
                : (kda ? delta_conventional_kernel<128, float, true> : delta_conventional_kernel<128, float, false>);
  else
    kern = in16 ? (kda ? delta_conventional_kernel<64, bf16, true> : delta_conventional_kernel<64, bf16, false>)
                : (kda ? delta_conventional_kernel<64, float, true> : delta_conventional_kernel<64, float, false>);
  kern<<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace rs
