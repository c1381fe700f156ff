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
#include <cstdlib>

#include "common.cuh"
#include "launch.h"
#include "mamba2_step.cuh"
#include "stream.cuh"

namespace rs {
namespace {

// ---------------------------------------------------------------- prep

constexpr int kPrepWarps = 8;   // warps per prep block
constexpr int kPrepDepth = 2;   // heads in flight per warp

struct M2Prep {
  int batch, H, G, P, W;
  const float* A;
  const float* D;
  const void* x;
  const void* B;
  const void* C;
  const float* dt;
  void* ring_x;
  void* ring_B;
  void* ring_C;
  float* ring_dt;
  int32_t* head;
  int32_t* len;
  int32_t* status;
  int32_t* sync;
  float* work;     // [b, H, wrow]: buffer terms [0, P), decay at P
  int wrow;
  int32_t* flags;  // [b]
};

// Shared memory of one prep warp (byte offsets): kPrepDepth head stages
// (buffered x rows in entry order, current x, ring dt row, dt/A/D) and the
// warp's cache for the current (sequence, group): C, B of the token, C.B_j.
struct M2PrepSmem {
  size_t hdr, xr, xt, dtr, sc, stage, Cf, Bt, CB, warp_bytes;
  __host__ __device__ M2PrepSmem(int P, int N, int W, int ti) {
    hdr = 0;                             // len, head, ok, seq as the issue side read them
    xr = 16;
    xt = xr + align_up((size_t)W * P * ti, 16);
    dtr = xt + align_up((size_t)P * ti, 16);
    sc = dtr + (size_t)ring_wd(W) * 4;   // dt, A, D of the head
    stage = align_up(sc + 16, 16);
    Cf = (size_t)kPrepDepth * stage;
    Bt = Cf + (size_t)N * 4;
    CB = Bt + align_up((size_t)N * ti, 16);
    warp_bytes = align_up(CB + (size_t)(W + 1) * 4, 128);
  }
};

// Preparation of a Mamba-2 decode. Each warp owns a contiguous range of
// heads (flat index seq * H + h) and walks it as a pipeline: async copies of
// a head's inputs (its buffered x rows, ring dt row, current x, dt, A, D) go
// out kPrepDepth heads ahead, so that many heads are in flight per SM. Per
// head, with dA_i = exp(dt_i A_h) over the n = len + 1 entries (entry len is
// the current token):
//   decay   = prod_i dA_i = exp(A_h sum_i dt_i)
//   w_j     = dt_j exp(A_h sum_{i>j} dt_i)
//   extra_p = sum_j w_j (C . B_j) x_j[p] + D_h x[p]
// go to work[seq, h] (extra in [0, P), decay at P); C.B_j is computed once
// per (sequence, group) of the warp. The warp then appends the head's token
// to the ring, and arrives once per sequence on its arrival counter; the
// last arrival bumps len. A sequence whose ring is full (or whose pointers
// are out of range) gets a status bit and flags[seq] = 0 and is untouched.
// PT is the head dimension P when known at compile time (0: runtime P).
template <int N, int PT, typename TI>
__global__ void __launch_bounds__(32 * kPrepWarps) mamba2_prep_kernel(const M2Prep a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int kNL = N / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int H = a.H, G = a.G, W = a.W, hpg = H / G;
  const int P = PT ? PT : a.P;
  const int Wd = ring_wd(W);
  const M2PrepSmem L(P, N, W, sizeof(TI));
  unsigned char* wbase = smem + (size_t)warp * L.warp_bytes;
  griddep_launch_dependents();  // the stream kernel may start streaming state rows
  const long long heads = (long long)a.batch * H;
  const long long nw = (long long)gridDim.x * kPrepWarps;
  const long long gw = (long long)blockIdx.x * kPrepWarps + warp;
  const int v0 = (int)(heads * gw / nw), v1 = (int)(heads * (gw + 1) / nw);
  if (v0 >= v1) return;
  const TI* xin = reinterpret_cast<const TI*>(a.x);
  const TI* Bin = reinterpret_cast<const TI*>(a.B);
  const TI* Cin = reinterpret_cast<const TI*>(a.C);
  const TI* rB = reinterpret_cast<const TI*>(a.ring_B);
  const int row = P * (int)sizeof(TI);  // bytes of one x row
  const int cpr = row / 16;             // 16-byte chunks per row
  // lane -> (row within a pass, chunk) for the row copies when cpr divides 32
  const bool lane_map = (32 % cpr) == 0;
  const int lrow = lane / cpr, lchunk = lane - (lane / cpr) * cpr, rstep = 32 / cpr;
  float* Cf = reinterpret_cast<float*>(wbase + L.Cf);
  TI* Btc = reinterpret_cast<TI*>(wbase + L.Bt);
  float* CB = reinterpret_cast<float*>(wbase + L.CB);
  const unsigned char* ringx = reinterpret_cast<const unsigned char*>(a.ring_x);

  // ---- issue side: (sequence, head) of the next head to fetch
  int i_seq = v0 / H, i_h = v0 - (v0 / H) * H;
  int i_len = 0, i_hd = 0;
  bool i_ok = false;
  int i_loaded = -1;  // sequence whose pointers the issue side holds
  int i_t = 0;        // next head (offset from v0) to fetch
  auto issue = [&]() {
    if (i_seq != i_loaded) {
      int l = 0, hh = 0;
      if (lane == 0) {
        l = a.len[i_seq];
        hh = a.head[i_seq];
      }
      i_len = __shfl_sync(kFull, l, 0);
      i_hd = __shfl_sync(kFull, hh, 0);
      i_ok = pointers_ok(i_hd, i_len, W) && i_len + 1 <= W;
      i_loaded = i_seq;
    }
    const int v = v0 + i_t;
    unsigned char* st = wbase + (size_t)(i_t % kPrepDepth) * L.stage;
    if (lane == 0) {
      int* hdr = reinterpret_cast<int*>(st + L.hdr);
      hdr[0] = i_len;
      hdr[1] = i_hd;
      hdr[2] = i_ok ? 1 : 0;
    }
    if (i_ok) {
      const unsigned char* xs = ringx + (size_t)v * W * row;
      if (lane_map) {
        for (int j = lrow; j < i_len; j += rstep) {
          const int slot = i_hd + j < W ? i_hd + j : i_hd + j - W;
          cp_async16(st + L.xr + j * row + lchunk * 16, xs + slot * row + lchunk * 16);
        }
      } else {
        for (int idx = lane; idx < i_len * cpr; idx += 32) {
          const int j = idx / cpr, c = idx - j * cpr;
          const int slot = i_hd + j < W ? i_hd + j : i_hd + j - W;
          cp_async16(st + L.xr + j * row + c * 16, xs + slot * row + c * 16);
        }
      }
      for (int c = lane; c < cpr; c += 32)
        cp_async16(st + L.xt + c * 16, reinterpret_cast<const unsigned char*>(xin) + (size_t)v * row + c * 16);
      if (lane < Wd / 4) cp_async16(st + L.dtr + lane * 16, a.ring_dt + (size_t)v * Wd + 4 * lane);
      float* sc = reinterpret_cast<float*>(st + L.sc);
      if (lane == 0) cp_async4(sc, a.dt + v);
      if (lane == 1) cp_async4(sc + 1, a.A + i_h);
      if (lane == 2) cp_async4(sc + 2, a.D + i_h);
    }
    cp_async_commit();  // one group per head (possibly empty)
    ++i_t;
    if (++i_h == H) {
      i_h = 0;
      ++i_seq;
    }
  };

  // ---- compute side
  int cur_seq = -1, len = 0, hd = 0;
  bool ok = false;
  int cb_seq = -1, cb_g = -1;  // (sequence, group) whose C.B_j the cache holds
  int seq_first = v0;          // first head of the current sequence in this range
  int seq = v0 / H, h = v0 - (v0 / H) * H;
  int g = h / hpg, hg = h - g * hpg;  // group of head h and h's index in it
  const int nv = v1 - v0;
  while (i_t < kPrepDepth - 1 && i_t < nv) issue();
  for (int t = 0; t < nv; ++t) {
    if (i_t < nv) {
      issue();
      cp_async_wait_group<kPrepDepth - 1>();  // head t has landed
    } else {
      cp_async_wait_all();  // the last heads of the range
    }
    __syncwarp();
    const int v = v0 + t;
    if (seq != cur_seq) {
      if (cur_seq >= 0 && ok && lane == 0)  // leaving a sequence: arrive with its heads
        arrive_and_finish(a.sync + cur_seq, v - seq_first, H, [&] { a.len[cur_seq] = len + 1; });
      const int* hdr = reinterpret_cast<const int*>(wbase + (size_t)(t % kPrepDepth) * L.stage + L.hdr);
      len = hdr[0];
      hd = hdr[1];
      ok = (hdr[2] & 1) != 0;
      cur_seq = seq;
      seq_first = v;
      if (h == 0 && lane == 0) {
        a.flags[seq] = ok ? 1 : 0;
        if (!ok)
          atomicOr(a.status + seq, pointers_ok(hd, len, W) ? REPLAYSSM_SEQ_RING_FULL
                                                           : REPLAYSSM_SEQ_BAD_POINTER);
      }
    }
    if (ok) {
      const unsigned char* st = wbase + (size_t)(t % kPrepDepth) * L.stage;
      // C.B_j of this (sequence, group), entries 0..len (entry len: the token)
      if (seq != cb_seq || g != cb_g) {
        cb_seq = seq;
        cb_g = g;
        float cf[kNL];
#pragma unroll
        for (int q = 0; q < kNL; ++q) {
          cf[q] = to_f(Cin[((size_t)seq * G + g) * N + lane + 32 * q]);
          Cf[lane + 32 * q] = cf[q];
        }
        for (int c = lane; c < N; c += 32) Btc[c] = Bin[((size_t)seq * G + g) * N + c];
        for (int j0 = 0; j0 <= len; j0 += 16) {
          float vv[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int j = min(j0 + q, len);
            const int slot = hd + j < W ? hd + j : hd + j - W;
            const TI* Bj = j < len ? rB + (((size_t)seq * W + slot) * G + g) * N
                                   : Bin + ((size_t)seq * G + g) * N;
            float pp = 0.f;
#pragma unroll
            for (int k = 0; k < kNL; ++k) pp = fmaf(cf[k], to_f(Bj[lane + 32 * k]), pp);
            vv[q] = pp;
          }
          float tot = reduce_scatter<16>(vv, lane);
          tot += __shfl_xor_sync(kFull, tot, 16);
          const int j = j0 + (lane & 15);
          if (lane < 16 && j <= len) CB[j] = tot;
        }
        __syncwarp();
      }
      // weights: lane j holds entries j and j + 32
      const float* dtr = reinterpret_cast<const float*>(st + L.dtr);
      const float* sc = reinterpret_cast<const float*>(st + L.sc);
      const float dt_tok = sc[0], Ah = sc[1], Dh = sc[2];
      const int n = len + 1;
      float dtv0, dtv1 = 0.f, cbv0, cbv1 = 0.f;
      {
        const int slot = hd + lane < W ? hd + lane : hd + lane - W;
        dtv0 = lane < len ? dtr[slot] : (lane == len ? dt_tok : 0.f);
        cbv0 = lane < n ? CB[lane] : 0.f;
      }
      if (n > 32) {
        const int j = lane + 32;
        const int slot = hd + j < W ? hd + j : hd + j - W;
        dtv1 = j < len ? dtr[slot] : (j == len ? dt_tok : 0.f);
        cbv1 = j < n ? CB[j] : 0.f;
      }
      float inc0 = dtv0, inc1 = dtv1;  // inclusive suffix sums of dt
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float tt = __shfl_down_sync(kFull, inc0, o);
        if (lane + o < 32) inc0 += tt;
      }
      if (n > 32) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float tt = __shfl_down_sync(kFull, inc1, o);
          if (lane + o < 32) inc1 += tt;
        }
        inc0 += __shfl_sync(kFull, inc1, 0);
      }
      const float total = __shfl_sync(kFull, inc0, 0);
      // exponents lie in [A_h sum dt, 0]; the fast exponential's relative
      // error (about 1e-6 there) is far inside the output tolerance
      const float w0 = dtv0 * __expf(Ah * (inc0 - dtv0)) * cbv0;
      const float w1 = n > 32 ? dtv1 * __expf(Ah * (inc1 - dtv1)) * cbv1 : 0.f;
      // buffer terms: lane owns rows p = 2 lane + {0, 1} (+ 64 k)
      const TI* xr = reinterpret_cast<const TI*>(st + L.xr);
      const TI* xt = reinterpret_cast<const TI*>(st + L.xt);
      const float c_tok = Dh + __shfl_sync(kFull, len < 32 ? w0 : w1, len & 31);
      float* wrow = a.work + (size_t)v * a.wrow;
#pragma unroll
      for (int p0 = 0; p0 < (PT ? PT : 256); p0 += 64) {  // every lane runs every iteration
        if (p0 >= P) break;
        const int p = p0 + 2 * lane;
        const bool act = p < P;
        float2 xv = act ? load2<TI>(xt + p) : make_float2(0.f, 0.f);
        float e0 = c_tok * xv.x, e1 = c_tok * xv.y;
        int j = 0;
        for (; j < len && j < 32; ++j) {
          const float c = __shfl_sync(kFull, w0, j);
          if (act) {
            xv = load2<TI>(xr + j * P + p);
            e0 = fmaf(c, xv.x, e0);
            e1 = fmaf(c, xv.y, e1);
          }
        }
        for (; j < len; ++j) {
          const float c = __shfl_sync(kFull, w1, j - 32);
          if (act) {
            xv = load2<TI>(xr + j * P + p);
            e0 = fmaf(c, xv.x, e0);
            e1 = fmaf(c, xv.y, e1);
          }
        }
        if (act) *reinterpret_cast<float2*>(wrow + p) = make_float2(e0, e1);
      }
      if (lane == 0) wrow[P] = __expf(Ah * total);
      // append the token: x row and dt of this head, B and C of its group
      const int slot = hd + len < W ? hd + len : hd + len - W;
      uint4* xd = reinterpret_cast<uint4*>(const_cast<unsigned char*>(ringx) +
                                           ((size_t)v * W + slot) * row);
      for (int c = lane; c < cpr; c += 32) xd[c] = reinterpret_cast<const uint4*>(xt)[c];
      if (lane == 0) a.ring_dt[(size_t)v * Wd + slot] = dt_tok;
      if (hg == 0) {
        TI* dB = reinterpret_cast<TI*>(a.ring_B) + (((size_t)seq * W + slot) * G + g) * N;
        for (int c = lane; c < N; c += 32) dB[c] = Btc[c];
        if (a.ring_C) {
          TI* dC = reinterpret_cast<TI*>(a.ring_C) + (((size_t)seq * W + slot) * G + g) * N;
          for (int c = lane; c < N; c += 32) dC[c] = Cin[((size_t)seq * G + g) * N + c];
        }
      }
      __syncwarp();
    }
    if (++hg == hpg) {
      hg = 0;
      ++g;
    }
    if (++h == H) {
      h = 0;
      g = 0;
      ++seq;
    }
  }
  cp_async_wait_all();
  if (cur_seq >= 0 && ok && lane == 0)
    arrive_and_finish(a.sync + cur_seq, v1 - seq_first, H, [&] { a.len[cur_seq] = len + 1; });
}

// ------------------------------------------------- fused step: coefficients

constexpr int kCoefWarps = 8;   // warps per coefficient block
constexpr int kCoefHeads = 8;   // heads per warp

struct M2Coef {
  int batch, H, G, W;
  const float* A;
  const float* D;
  const void* B;      // token inputs [b, G, N]
  const void* C;
  const float* dt;    // [b, H]
  void* ring_B;
  void* ring_C;
  float* ring_dt;
  const int32_t* head;
  const int32_t* len;
  int32_t* status;
  float* work;   // [b, H, kStepRow]
  float* bfold;  // [b, G, kStepMaxW, N]
};

// Per-head coefficients of the fused fold + decode step. A sequence whose
// ring is full (len + 1 > W) is folded first: its nf = len entries leave the
// ring (head += nf, len = 0) and the token is decoded after them. The decode
// then replays the ld buffered entries (ld = len without a fold, 0 with one)
// and the token, entry ld; with dA_i = exp(dt_i A_h) over those entries:
//   c_j    = w_j (C . B_j),  w_j = dt_j exp(A_h sum_{i>j} dt_i),  j < ld
//   c_tok  = dt_tok (C . B_tok) + D_h
//   decay  = exp(A_h sum_i dt_i)
// and for a fold, over its nf entries, the fold weights w_j and the fold
// decay exp(A_h sum_j dt_j). The stream kernel computes the buffer terms
// sum_j c_j x_j[p] + c_tok x[p] itself from the ring x rows, so this grid
// reads no x at all and is short: its dependent stream kernel starts as it
// ends (or earlier, on SMs it leaves).
//
// One warp per (sequence, chunk of kCoefHeads heads); half-warps take one
// head each, lane j of a half holding entry j. The warp is latency-bound, so
// it issues every load it needs (C, the B rows, and the dt rows, token dt, A
// and D of all its heads) before it computes or stores anything. C . B_j is
// computed once per group the chunk touches. The token's dt goes into the
// ring here, and the warp holding a group's first head copies the group's
// folded B rows out as floats and then appends the token's B and C. The x
// row of the token is appended by the stream kernel, row by row, after it
// has read the ring. No slot this grid writes is one it, or any other warp
// of the grid, reads: without a fold the token's slot is past the buffered
// entries, and with one only the writing warp reads the old entries, first.
template <int N, typename TI>
__global__ void __launch_bounds__(32 * kCoefWarps, 2) mamba2_step_coef_kernel(const M2Coef a) {
  constexpr int E = N / 32;                   // B and C elements per lane
  constexpr int kPasses = kCoefHeads / 2;     // heads per half-warp
  constexpr int kMaxG = kCoefHeads;           // groups a chunk can touch
  griddep_launch_dependents();  // the stream kernel may start streaming state rows
  const int lane = threadIdx.x & 31;
  const int H = a.H, G = a.G, W = a.W, hpg = H / G, Wd = ring_wd(W);
  const int nch = (H + kCoefHeads - 1) / kCoefHeads;
  const long long wv = (long long)blockIdx.x * kCoefWarps + (threadIdx.x >> 5);
  if (wv >= (long long)a.batch * nch) return;
  const int seq = (int)(wv / nch);
  const int h0 = (int)(wv - (long long)seq * nch) * kCoefHeads, h1 = min(h0 + kCoefHeads, H);
  int l = 0, hh = 0;
  if (lane == 0) {
    l = a.len[seq];
    hh = a.head[seq];
  }
  const int len = __shfl_sync(kFull, l, 0), hd = __shfl_sync(kFull, hh, 0);
  if (!pointers_ok(hd, len, W)) {
    if (h0 == 0 && lane == 0) atomicOr(a.status + seq, REPLAYSSM_SEQ_BAD_POINTER);
    return;
  }
  const int nf = len + 1 > W ? len : 0;     // entries folded before the token
  const int hdd = nf ? (hd + len) % W : hd;  // ring head of the decode
  const int ld = nf ? 0 : len;              // buffered entries the decode replays
  auto slot_of = [W](int s) { return s < W ? s : s - W; };
  const int tslot = slot_of(hdd + ld);      // the token's slot
  const TI* Bin = reinterpret_cast<const TI*>(a.B);
  const TI* Cin = reinterpret_cast<const TI*>(a.C);
  const TI* rB = reinterpret_cast<const TI*>(a.ring_B);
  const int half = lane >> 4, j = lane & 15;
  const int g0 = h0 / hpg, ng = (h1 - 1) / hpg - g0 + 1;  // groups of the chunk

  // ---- every load first: per pass (head h0 + 2 p + half) this lane's decode
  // dt, fold dt, and the head's token dt, A and D
  float dd[kPasses], fd[kPasses], dtt[kPasses], Av[kPasses], Dv[kPasses];
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int h = min(h0 + 2 * p + half, h1 - 1);
    const size_t v = (size_t)seq * H + h;
    const float* rdt = a.ring_dt + v * Wd;
    dd[p] = j < ld ? rdt[slot_of(hdd + j)] : 0.f;
    fd[p] = j < nf ? rdt[slot_of(hd + j)] : 0.f;
    dtt[p] = a.dt[v];
    Av[p] = a.A[h];
    Dv[p] = a.D[h];
  }
  // C . B_j of each group of the chunk for the decode's entries 0..ld (entry
  // ld: the token); lane l ends with entry l & 15 (ld < kStepMaxW = 16).
  float cbv[kMaxG];
#pragma unroll
  for (int gl = 0; gl < kMaxG; ++gl) {
    cbv[gl] = 0.f;
    if (gl >= ng) continue;
    const int g = g0 + gl;
    float cf[E];
    load_vec<TI, E>(Cin + ((size_t)seq * G + g) * N + lane * E, cf);
    Raw<TI, E> bv[kStepMaxW];
#pragma unroll
    for (int q = 0; q < kStepMaxW; ++q) {
      if (q <= ld) {
        const TI* Bj = q < ld ? rB + (((size_t)seq * W + slot_of(hdd + q)) * G + g) * N
                              : Bin + ((size_t)seq * G + g) * N;
        load_raw<TI, E>(Bj + lane * E, bv[q]);
      }
    }
    float vv[kStepMaxW];
#pragma unroll
    for (int q = 0; q < kStepMaxW; ++q) {
      float pp = 0.f;
      if (q <= ld) {
        float bf[E];
        raw_to_f<TI, E>(bv[q], bf);
#pragma unroll
        for (int e = 0; e < E; ++e) pp = fmaf(cf[e], bf[e], pp);
      }
      vv[q] = pp;
    }
    const float tot = reduce_scatter<kStepMaxW>(vv, lane);
    cbv[gl] = tot + __shfl_xor_sync(kFull, tot, 16);
  }

  // ---- weights, one head per half-warp and pass
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int h = h0 + 2 * p + half;
    if (h0 + 2 * p >= h1) break;  // warp-uniform
    const bool act = h < h1;
    const size_t v = (size_t)seq * H + (act ? h : h1 - 1);
    float cb = 0.f;
#pragma unroll
    for (int gl = 0; gl < kMaxG; ++gl)
      if (gl == (act ? h : h1 - 1) / hpg - g0) cb = cbv[gl];
    // decode weights: inclusive suffix sums of dt over the half's 16 lanes
    const float d = j == ld ? dtt[p] : dd[p];
    float sfx = d;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const float t = __shfl_down_sync(kFull, sfx, o, 16);
      if (j + o < 16) sfx += t;
    }
    const float total = __shfl_sync(kFull, sfx, 0, 16);
    // exponents lie in [A_h sum dt, 0]; the fast exponential's relative
    // error (about 1e-6 there) is far inside the output tolerance
    const float c = d * __expf(Av[p] * (sfx - d)) * cb;
    float* wr = a.work + v * kStepRow;
    if (act) {
      wr[j] = j < ld ? c : 0.f;
      if (j == ld) wr[kStepTok] = c + Dv[p];
      if (j == 0) wr[kStepDecay] = __expf(Av[p] * total);
    }
    if (nf) {  // fold weights over the nf entries from the old head
      const float f = fd[p];
      float fs = f;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        const float t = __shfl_down_sync(kFull, fs, o, 16);
        if (j + o < 16) fs += t;
      }
      const float ftot = __shfl_sync(kFull, fs, 0, 16);
      if (act) {
        wr[kStepFoldW + j] = j < nf ? f * expf(Av[p] * (fs - f)) : 0.f;
        if (j == 0) wr[kStepFoldDecay] = expf(Av[p] * ftot);
      }
    }
    // the token's dt, after the half has read the row (every load of it was
    // consumed above); with a fold its slot is entry 0's
    if (act && j == 0) a.ring_dt[v * Wd + tslot] = dtt[p];
  }

  // ---- groups whose first head is in this chunk: folded B rows (all loads
  // first), then the token's B and C
  for (int g = g0; g * hpg < h1; ++g) {
    if (g * hpg < h0) continue;
    const size_t gi = (size_t)seq * G + g;
    if (nf) {
      Raw<TI, E> bq[kStepMaxW];
#pragma unroll
      for (int jj = 0; jj < kStepMaxW; ++jj)
        if (jj < nf) load_raw<TI, E>(rB + (((size_t)seq * W + slot_of(hd + jj)) * G + g) * N + lane * E, bq[jj]);
      float* Bs = a.bfold + gi * kStepMaxW * N + lane * E;
#pragma unroll
      for (int jj = 0; jj < kStepMaxW; ++jj) {
        if (jj < nf) {
          float bf[E];
          raw_to_f<TI, E>(bq[jj], bf);
#pragma unroll
          for (int e = 0; e < E; ++e) Bs[(size_t)jj * N + e] = bf[e];
        }
      }
      __syncwarp();
    }
    TI* dB = reinterpret_cast<TI*>(a.ring_B) + (((size_t)seq * W + tslot) * G + g) * N;
    for (int cc = lane; cc < N; cc += 32) dB[cc] = Bin[gi * N + cc];
    if (a.ring_C) {
      TI* dC = reinterpret_cast<TI*>(a.ring_C) + (((size_t)seq * W + tslot) * G + g) * N;
      for (int cc = lane; cc < N; cc += 32) dC[cc] = Cin[gi * N + cc];
    }
  }
}

// -------------------------------------------------------------- verify prep

struct M2VPrep {
  int batch, H, G, P, W, K;
  const float* A;
  const float* D;
  const void* x;       // drafts [b, K, H, P]
  const void* B;       // [b, K, G, N]
  const void* C;       // [b, K, G, N]
  const float* dt;     // [b, K, H]
  void* ring_x;
  void* ring_B;
  void* ring_C;
  float* ring_dt;
  int32_t* head;
  int32_t* len;
  int32_t* status;
  float* work;         // [b, K, H, wrow]: buffer terms [0, P), decay at P
  int wrow;
  int32_t* flags;      // [b]
};

// Preparation of a Mamba-2 speculative verify, one warp per head. Entry
// j < len is ring slot (head + j) mod W; entry len + i is draft i. For draft
// i (entries 0..len + i visible), with dA_l = exp(dt_l A_h):
//   decay_i    = prod_{l <= len+i} dA_l
//   extra_i[p] = sum_{j <= len+i} dt_j prod_{j < l <= len+i} dA_l (C_i . B_j) x_j[p] + D_h x_i[p]
// go to work row (seq, i, h). The drafts are appended at slots
// (head + len + i) mod W; len is unchanged (accept moves it). A sequence
// without room for K drafts gets a status bit and flags[seq] = 0.
template <int N, typename TI>
__global__ void __launch_bounds__(256) mamba2_verify_prep_kernel(const M2VPrep a) {
  constexpr int kNL = N / 32;
  const int lane = threadIdx.x & 31;
  const int H = a.H, G = a.G, P = a.P, W = a.W, K = a.K, hpg = H / G, Wd = ring_wd(W);
  const long long heads = (long long)a.batch * H;
  const long long nw = (long long)gridDim.x * (blockDim.x >> 5);
  const TI* xin = reinterpret_cast<const TI*>(a.x);
  const TI* Bin = reinterpret_cast<const TI*>(a.B);
  const TI* Cin = reinterpret_cast<const TI*>(a.C);
  const TI* rB = reinterpret_cast<const TI*>(a.ring_B);
  const TI* rx = reinterpret_cast<const TI*>(a.ring_x);
  griddep_launch_dependents();  // the stream kernel may start streaming state rows
  for (long long v = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); v < heads; v += nw) {
    const int seq = (int)(v / H), h = (int)(v - (long long)seq * H), g = h / hpg;
    int l = 0, hh = 0;
    if (lane == 0) {
      l = a.len[seq];
      hh = a.head[seq];
    }
    const int len = __shfl_sync(kFull, l, 0), hd = __shfl_sync(kFull, hh, 0);
    const bool ok = pointers_ok(hd, len, W) && len + K <= W;
    if (h == 0 && lane == 0) {
      a.flags[seq] = ok ? 1 : 0;
      if (!ok)
        atomicOr(a.status + seq, pointers_ok(hd, len, W) ? REPLAYSSM_SEQ_RING_FULL
                                                         : REPLAYSSM_SEQ_BAD_POINTER);
    }
    if (!ok) continue;
    const float Ah = a.A[h], Dh = a.D[h];
    auto slot_of = [&](int j) { return hd + j < W ? hd + j : hd + j - W; };
    auto entry_dt = [&](int j) -> float {
      if (j < len) return a.ring_dt[(size_t)v * Wd + slot_of(j)];
      if (j < len + K) return a.dt[((size_t)seq * K + (j - len)) * H + h];
      return 0.f;
    };
    auto entry_B = [&](int j) -> const TI* {
      return j < len ? rB + (((size_t)seq * W + slot_of(j)) * G + g) * N
                     : Bin + (((size_t)seq * K + (j - len)) * G + g) * N;
    };
    auto entry_x = [&](int j) -> const TI* {
      return j < len ? rx + ((size_t)v * W + slot_of(j)) * P
                     : xin + (((size_t)seq * K + (j - len)) * H + h) * P;
    };
    const float dtv0 = entry_dt(lane), dtv1 = entry_dt(lane + 32);
    for (int i = 0; i < K; ++i) {
      const int top = len + i;
      // C_i . B_j for entries 0..top: lane j holds entries j and j + 32
      float cf[kNL];
#pragma unroll
      for (int q = 0; q < kNL; ++q) cf[q] = to_f(Cin[(((size_t)seq * K + i) * G + g) * N + lane + 32 * q]);
      float cb0 = 0.f, cb1 = 0.f;
      for (int j0 = 0; j0 <= top; j0 += 16) {
        float vv[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const TI* Bj = entry_B(min(j0 + q, top));
          float pp = 0.f;
#pragma unroll
          for (int k = 0; k < kNL; ++k) pp = fmaf(cf[k], to_f(Bj[lane + 32 * k]), pp);
          vv[q] = pp;
        }
        float tot = reduce_scatter<16>(vv, lane);
        tot += __shfl_xor_sync(kFull, tot, 16);  // every lane: entry j0 + (lane & 15)
        const float t0 = __shfl_sync(kFull, tot, (lane - j0) & 15);
        const float t1 = __shfl_sync(kFull, tot, (lane + 32 - j0) & 15);
        if (lane >= j0 && lane < j0 + 16) cb0 = t0;
        if (lane + 32 >= j0 && lane + 32 < j0 + 16) cb1 = t1;
      }
      // weights from suffix sums of dt over entries 0..top
      const float d0 = lane <= top ? dtv0 : 0.f, d1 = lane + 32 <= top ? dtv1 : 0.f;
      float inc0 = d0, inc1 = d1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t0 = __shfl_down_sync(kFull, inc0, o), t1 = __shfl_down_sync(kFull, inc1, o);
        if (lane + o < 32) {
          inc0 += t0;
          inc1 += t1;
        }
      }
      inc0 += __shfl_sync(kFull, inc1, 0);
      const float total = __shfl_sync(kFull, inc0, 0);
      float c0 = lane <= top ? d0 * __expf(Ah * (inc0 - d0)) * cb0 : 0.f;
      float c1 = lane + 32 <= top ? d1 * __expf(Ah * (inc1 - d1)) * cb1 : 0.f;
      if (lane == top) c0 += Dh;
      if (lane + 32 == top) c1 += Dh;
      float* wrow = a.work + (((size_t)seq * K + i) * H + h) * a.wrow;
      for (int p0 = 0; p0 < P; p0 += 64) {  // every lane runs every iteration
        const int p = p0 + 2 * lane;
        const bool act = p < P;
        float e0 = 0.f, e1 = 0.f;
        for (int j = 0; j <= top; ++j) {
          const float c = __shfl_sync(kFull, j < 32 ? c0 : c1, j & 31);
          if (act) {
            const float2 xv = load2<TI>(entry_x(j) + p);
            e0 = fmaf(c, xv.x, e0);
            e1 = fmaf(c, xv.y, e1);
          }
        }
        if (act) *reinterpret_cast<float2*>(wrow + p) = make_float2(e0, e1);
      }
      if (lane == 0) wrow[P] = __expf(Ah * total);
    }
    // append the drafts: x rows and dt of this head, B and C of its group
    for (int i = 0; i < K; ++i) {
      const int slot = slot_of(len + i);
      const size_t xb = (size_t)P * sizeof(TI);
      block_copy_warp(reinterpret_cast<unsigned char*>(a.ring_x) + ((size_t)v * W + slot) * xb,
                      reinterpret_cast<const unsigned char*>(xin) + (((size_t)seq * K + i) * H + h) * xb,
                      (int)xb, lane);
      if (lane == 0) a.ring_dt[(size_t)v * Wd + slot] = a.dt[((size_t)seq * K + i) * H + h];
      if (h - g * hpg == 0) {
        const size_t src = (((size_t)seq * K + i) * G + g) * N, dst = (((size_t)seq * W + slot) * G + g) * N;
        for (int c = lane; c < N; c += 32) reinterpret_cast<TI*>(a.ring_B)[dst + c] = Bin[src + c];
        if (a.ring_C)
          for (int c = lane; c < N; c += 32) reinterpret_cast<TI*>(a.ring_C)[dst + c] = Cin[src + c];
      }
    }
  }
}

constexpr int kFoldThreads = 256;
constexpr int kFoldRows = 8;  // contiguous state rows per thread (loads in flight)

struct M2Fold {
  int batch, H, G, P, W, HB, k_next, force;  // HB: heads per unit
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

// Shared memory of the fold block (byte offsets).
struct M2FoldSmem {
  size_t xr, Br, dtr, Av, coef, Bf, wts, dec, total;
  __host__ __device__ M2FoldSmem(int HB, int P, int N, int W, int ti) {
    xr = 0;                                                  // [HB][W][P] x_j (in_dtype)
    Br = align_up((size_t)HB * W * P * ti, 16);              // [W][N] B_j (in_dtype)
    dtr = Br + align_up((size_t)W * N * ti, 16);             // [HB][Wd] ring dt rows
    Av = dtr + (size_t)HB * ring_wd(W) * 4;                  // [HB] A
    coef = Av + align_up((size_t)HB * 4, 16);                // [HB][W][P] w_j x_j[p]
    Bf = coef + (size_t)HB * W * P * 4;                      // [W][N] B_j as float
    wts = Bf + (size_t)W * N * 4;                            // [HB][W] w_j
    dec = wts + (size_t)HB * W * 4;                          // [HB] decay
    total = dec + (size_t)HB * 4;
  }
};

// Consolidate for Mamba-2. Units are (sequence, HB consecutive heads); only
// units of folding sequences do work (one parallel pre-scan of the pointers
// per block). For a unit with n = len buffered entries the fold is the
// rank-n update
//   h_new[p][c] = decay h[p][c] + sum_j coef[j][p] B_j[c],
//   coef[j][p] = w_j x_j[p],  w_j = dt_j exp(A sum_{i>j} dt_i),
//   decay = exp(A sum_i dt_i).
// The unit's ring rows are staged with async copies, then coef and B are
// expanded to float in shared memory. Each thread owns a tile of kFoldRows
// contiguous rows by one float4 of columns: per entry j it reads two float4
// of coef (the same address across the lanes of a row: a broadcast) and one
// float4 of B, and issues 32 FMAs. The FP32 checkpoint and its BF16 read copy
// are written once.
template <int N, typename TI>
__global__ void __launch_bounds__(kFoldThreads, 3) mamba2_fold_kernel(const M2Fold a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ FoldList fl;
  constexpr int CT = N / 4;              // lanes across a row (one float4 each)
  constexpr int SUB = 32 / CT;           // row tiles per warp
  constexpr int kWarps = kFoldThreads / 32;
  constexpr int kRowStep = kWarps * SUB * kFoldRows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c4 = lane % CT, sub = lane / CT;
  const int H = a.H, G = a.G, P = a.P, W = a.W, HB = a.HB, hpg = H / G, Wd = ring_wd(W);
  const int per_seq = (H + HB - 1) / HB;
  const M2FoldSmem L(HB, P, N, W, sizeof(TI));
  const TI* xr = reinterpret_cast<const TI*>(smem + L.xr);
  const TI* Br = reinterpret_cast<const TI*>(smem + L.Br);
  const float* dtr = reinterpret_cast<const float*>(smem + L.dtr);
  const float* Av = reinterpret_cast<const float*>(smem + L.Av);
  float* coef = reinterpret_cast<float*>(smem + L.coef);
  float* Bf = reinterpret_cast<float*>(smem + L.Bf);
  float* wts = reinterpret_cast<float*>(smem + L.wts);
  float* dec = reinterpret_cast<float*>(smem + L.dec);
  const unsigned char* rx = reinterpret_cast<const unsigned char*>(a.ring_x);
  const unsigned char* rB = reinterpret_cast<const unsigned char*>(a.ring_B);
  const int xrow = P * (int)sizeof(TI), xcpr = xrow / 16;  // x row bytes, 16 B chunks
  const int brow = N * (int)sizeof(TI), bcpr = brow / 16;  // B row bytes, chunks

  collect_folds(fl, (long long)a.batch * per_seq, per_seq, a.len, a.head, a.status, W, a.k_next,
                a.force);
  // B rows (entries 0..n-1) of group g of sequence seq, as float
  auto stage_B = [&](int seq, int g, int n, int hd) {
    for (int idx = tid; idx < n * bcpr; idx += kFoldThreads) {
      const int j = idx / bcpr, c = idx - j * bcpr;
      const int slot = hd + j < W ? hd + j : hd + j - W;
      cp_async16(smem + L.Br + (size_t)j * brow + c * 16,
                 rB + (((size_t)seq * W + slot) * G + g) * brow + c * 16);
    }
    cp_async_wait_all();
    __syncthreads();
    for (int i = tid; i < n * N; i += kFoldThreads) Bf[i] = to_f(Br[i]);
  };
  for (int f = 0; f < fl.count; ++f) {
    const int t = fl.tile[f], n = fl.len[f], hd = fl.head[f];
    const int seq = t / per_seq, h0 = (t - seq * per_seq) * HB, nh = min(HB, H - h0);
    // stage the unit's x rows, dt rows and A
    for (int idx = tid; idx < nh * n * xcpr; idx += kFoldThreads) {
      const int hh = idx / (n * xcpr), rem = idx - hh * (n * xcpr);
      const int j = rem / xcpr, c = rem - j * xcpr;
      const int slot = hd + j < W ? hd + j : hd + j - W;
      cp_async16(smem + L.xr + ((size_t)hh * W + j) * xrow + c * 16,
                 rx + (((size_t)seq * H + h0 + hh) * W + slot) * xrow + c * 16);
    }
    for (int idx = tid; idx < nh * Wd / 4; idx += kFoldThreads)
      cp_async16(smem + L.dtr + 16 * idx, a.ring_dt + ((size_t)seq * H + h0) * Wd + 4 * idx);
    for (int hh = tid; hh < nh; hh += kFoldThreads)
      cp_async4(smem + L.Av + 4 * hh, a.A + h0 + hh);
    int g_loaded = h0 / hpg;
    stage_B(seq, g_loaded, n, hd);  // waits for all copies above too
    // weights and decay, one thread per head
    for (int hh = tid; hh < nh; hh += kFoldThreads) {
      const float Ah = Av[hh];
      float acc = 0.f;
      for (int j = n - 1; j >= 0; --j) {
        const float dtj = dtr[hh * Wd + (hd + j < W ? hd + j : hd + j - W)];
        wts[hh * W + j] = dtj * expf(Ah * acc);
        acc += dtj;
      }
      dec[hh] = expf(Ah * acc);
    }
    __syncthreads();
    for (int i = tid; i < nh * n * P; i += kFoldThreads) {
      const int hh = i / (n * P), rem = i - hh * (n * P), j = rem / P;
      coef[(size_t)hh * W * P + rem] = wts[hh * W + j] * to_f(xr[(size_t)hh * W * P + rem]);
    }
    __syncthreads();
    for (int hh = 0; hh < nh; ++hh) {
      const int g = (h0 + hh) / hpg;
      if (g != g_loaded) {  // B rows of this head's group
        __syncthreads();
        stage_B(seq, g, n, hd);
        __syncthreads();
        g_loaded = g;
      }
      const float decay = dec[hh];
      const float* ch = coef + (size_t)hh * W * P;
      float4* St = reinterpret_cast<float4*>(a.S + ((size_t)seq * H + h0 + hh) * P * N);
      uint2* Rt = a.Sr ? reinterpret_cast<uint2*>(a.Sr + ((size_t)seq * H + h0 + hh) * P * N) : nullptr;
      for (int p0 = (warp * SUB + sub) * kFoldRows; p0 < P; p0 += kRowStep) {
        float4 acc[kFoldRows];
#pragma unroll
        for (int r = 0; r < kFoldRows; ++r) {
          const float4 hv = St[(size_t)(p0 + r) * CT + c4];
          acc[r] = make_float4(decay * hv.x, decay * hv.y, decay * hv.z, decay * hv.w);
        }
#pragma unroll 2
        for (int j = 0; j < n; ++j) {
          const float4 b = reinterpret_cast<const float4*>(Bf + j * N)[c4];
          const float4 cl = reinterpret_cast<const float4*>(ch + j * P + p0)[0];
          const float4 ch4 = reinterpret_cast<const float4*>(ch + j * P + p0)[1];
          const float cr[kFoldRows] = {cl.x, cl.y, cl.z, cl.w, ch4.x, ch4.y, ch4.z, ch4.w};
#pragma unroll
          for (int r = 0; r < kFoldRows; ++r) {
            acc[r].x = fmaf(cr[r], b.x, acc[r].x);
            acc[r].y = fmaf(cr[r], b.y, acc[r].y);
            acc[r].z = fmaf(cr[r], b.z, acc[r].z);
            acc[r].w = fmaf(cr[r], b.w, acc[r].w);
          }
        }
#pragma unroll
        for (int r = 0; r < kFoldRows; ++r) {
          St[(size_t)(p0 + r) * CT + c4] = acc[r];
          if (Rt)
            Rt[(size_t)(p0 + r) * CT + c4] =
                make_uint2(pack_bf16x2(acc[r].x, acc[r].y), pack_bf16x2(acc[r].z, acc[r].w));
        }
      }
    }
    __syncthreads();
    if (tid == 0)
      arrive_and_finish(a.sync + seq, nh, H, [&] {
        a.head[seq] = (hd + n) % W;
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

}  // namespace

namespace {

// Launches the preparation kernel of the plain decode.
cudaError_t launch_prep(const replayssm_dims& d, const M2Prep& p, cudaStream_t st) {
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  const int ti = in16 ? 2 : 4;
  const M2PrepSmem L(d.dv, d.dk, d.window, ti);
  const size_t smem = L.warp_bytes * kPrepWarps;
  const long long heads = (long long)d.batch * d.heads;
  // as many resident warps as shared memory allows (latency-bound work)
  const int per_sm = std::max(1, std::min(8, (int)(device_info().smem_optin / (smem + 1024))));
  const long long grid = std::min<long long>((heads + kPrepWarps - 1) / kPrepWarps,
                                             (long long)device_info().sms * per_sm);
  cudaError_t e;
#define RS_PREP(N_, PT_, TI_)                                                                   \
  {                                                                                            \
    auto k = mamba2_prep_kernel<N_, PT_, TI_>;                                                 \
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);       \
    if (e != cudaSuccess) return e;                                                            \
    k<<<(unsigned)grid, 32 * kPrepWarps, smem, st>>>(p);                                       \
  }
#define RS_PREP_P(N_, TI_)                                                                      \
  if (d.dv == 64) RS_PREP(N_, 64, TI_) else if (d.dv == 128) RS_PREP(N_, 128, TI_) else RS_PREP(N_, 0, TI_)
  if (d.dk == 128) {
    if (in16) { RS_PREP_P(128, bf16) } else { RS_PREP_P(128, float) }
  } else {
    if (in16) { RS_PREP_P(64, bf16) } else { RS_PREP_P(64, float) }
  }
#undef RS_PREP_P
#undef RS_PREP
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mamba2_decode(const replayssm_dims& d, const replayssm_state& s, const float* A,
                                 const float* D, const void* x, const void* B, const void* C,
                                 const float* dt, float* y, cudaStream_t st) {
  const WorkLayout wl(d, 1);
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  M2Prep p{d.batch, d.heads, d.groups, d.dv, d.window, A, D, x, B, C, dt,
           s.ring_x, s.ring_B, s.ring_C, s.ring_dt, s.ring_head, s.ring_len, s.status, s.sync,
           s.work, wl.row, wl.flags(s.work)};
  cudaError_t e = launch_prep(d, p, st);
  if (e != cudaSuccess) return e;
  // Stream: y = decay * (S C) + extra, C straight from the token input.
  StreamArgs sa{};
  sa.batch = d.batch;
  sa.H = d.heads;
  sa.P = d.dv;
  sa.K = 1;
  sa.S = s.S_read ? (const void*)s.S_read : (const void*)s.S_ckpt;
  sa.out = y;
  sa.work = s.work;
  sa.wrow = wl.row;
  sa.vec_off = -1;
  sa.extra_off = 0;
  sa.scale_off = d.dv;
  sa.flags = wl.flags(s.work);
  sa.vin = C;
  sa.G = d.groups;
  sa.status = s.status;
  const bool rd16 = s.S_read != nullptr;
  if (d.dk == 128) {
    if (rd16) return in16 ? launch_stream<128, bf16, bf16, 1>(sa, st) : launch_stream<128, bf16, float, 1>(sa, st);
    return in16 ? launch_stream<128, float, bf16, 1>(sa, st) : launch_stream<128, float, float, 1>(sa, st);
  }
  if (rd16) return in16 ? launch_stream<64, bf16, bf16, 1>(sa, st) : launch_stream<64, bf16, float, 1>(sa, st);
  return in16 ? launch_stream<64, float, bf16, 1>(sa, st) : launch_stream<64, float, float, 1>(sa, st);
}

cudaError_t launch_mamba2_verify(const replayssm_dims& d, const replayssm_state& s, int K,
                                 const float* A, const float* D, const void* x, const void* B,
                                 const void* C, const float* dt, float* y, cudaStream_t st) {
  const WorkLayout wl(d, K);
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  M2VPrep p{d.batch, d.heads, d.groups, d.dv, d.window, K, A, D, x, B, C, dt,
            s.ring_x, s.ring_B, s.ring_C, s.ring_dt, s.ring_head, s.ring_len, s.status,
            s.work, wl.row, wl.flags(s.work)};
  const long long heads = (long long)d.batch * d.heads;
  const int grid = (int)std::min<long long>((heads + 7) / 8, (long long)device_info().sms * 8);
  if (d.dk == 128) {
    if (in16) mamba2_verify_prep_kernel<128, bf16><<<grid, 256, 0, st>>>(p);
    else mamba2_verify_prep_kernel<128, float><<<grid, 256, 0, st>>>(p);
  } else {
    if (in16) mamba2_verify_prep_kernel<64, bf16><<<grid, 256, 0, st>>>(p);
    else mamba2_verify_prep_kernel<64, float><<<grid, 256, 0, st>>>(p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // Stream: y_i = decay_i * (S C_i) + extra_i, C_i straight from the drafts.
  StreamArgs sa{};
  sa.batch = d.batch;
  sa.H = d.heads;
  sa.P = d.dv;
  sa.K = K;
  sa.S = s.S_read ? (const void*)s.S_read : (const void*)s.S_ckpt;
  sa.out = y;
  sa.work = s.work;
  sa.wrow = wl.row;
  sa.vec_off = -1;
  sa.extra_off = 0;
  sa.scale_off = d.dv;
  sa.flags = wl.flags(s.work);
  sa.vin = C;
  sa.G = d.groups;
  sa.status = s.status;
  const bool rd16 = s.S_read != nullptr;
#define RS_VSTREAM(KM_)                                                                        \
  if (d.dk == 128) {                                                                           \
    if (rd16) return in16 ? launch_stream<128, bf16, bf16, KM_>(sa, st) : launch_stream<128, bf16, float, KM_>(sa, st); \
    return in16 ? launch_stream<128, float, bf16, KM_>(sa, st) : launch_stream<128, float, float, KM_>(sa, st);       \
  }                                                                                            \
  if (rd16) return in16 ? launch_stream<64, bf16, bf16, KM_>(sa, st) : launch_stream<64, bf16, float, KM_>(sa, st);   \
  return in16 ? launch_stream<64, float, bf16, KM_>(sa, st) : launch_stream<64, float, float, KM_>(sa, st);
  if (K <= 4) {
    RS_VSTREAM(4)
  }
  RS_VSTREAM(8)
#undef RS_VSTREAM
}

cudaError_t launch_mamba2_fold(const replayssm_dims& d, const replayssm_state& s, const float* A,
                               int k_next, int force, cudaStream_t st) {
  // heads per unit: the staged rows and coefficients stay under 48 KB
  const int ti = d.in_dtype == REPLAYSSM_BF16 ? 2 : 4;
  int HB = 8;
  while (HB > 1 && (size_t)HB * d.window * d.dv * (ti + 4) > 48 * 1024) HB /= 2;
  M2Fold a{d.batch, d.heads, d.groups, d.dv, d.window, HB, k_next, force, s.S_ckpt,
           reinterpret_cast<bf16*>(s.S_read), A, s.ring_x, s.ring_B, s.ring_dt,
           s.ring_head, s.ring_len, s.status, s.sync};
  const long long units = (long long)d.batch * ((d.heads + HB - 1) / HB);
  const M2FoldSmem L(HB, d.dv, d.dk, d.window, ti);
  const int grid = std::max<long long>((units + kMaxFoldTiles - 1) / kMaxFoldTiles,
                                       std::min<long long>(units, (long long)device_info().sms * 3));
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  cudaError_t e;
  void (*kern)(const M2Fold);
  if (d.dk == 128)
    kern = in16 ? mamba2_fold_kernel<128, bf16> : mamba2_fold_kernel<128, float>;
  else
    kern = in16 ? mamba2_fold_kernel<64, bf16> : mamba2_fold_kernel<64, float>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
  if (e != cudaSuccess) return e;
  kern<<<grid, kFoldThreads, L.total, st>>>(a);
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

namespace {

// Launches the coefficient kernel of the fused step. Its blocks use no shared
// memory (and ask for the shared-memory carveout the stream kernel needs),
// so the stream kernel's blocks fit beside them and start at once.
cudaError_t launch_step_coef(const replayssm_dims& d, const M2Coef& p, cudaStream_t st) {
  const long long warps = (long long)d.batch * ((d.heads + kCoefHeads - 1) / kCoefHeads);
  const unsigned grid = (unsigned)((warps + kCoefWarps - 1) / kCoefWarps);
  void (*kern)(const M2Coef);
  if (d.dk == 128)
    kern = d.in_dtype == REPLAYSSM_BF16 ? mamba2_step_coef_kernel<128, bf16>
                                        : mamba2_step_coef_kernel<128, float>;
  else
    kern = d.in_dtype == REPLAYSSM_BF16 ? mamba2_step_coef_kernel<64, bf16>
                                        : mamba2_step_coef_kernel<64, float>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  kern<<<grid, 32 * kCoefWarps, 0, st>>>(p);
  return cudaGetLastError();
}

template <int N, typename TS, typename TV>
cudaError_t launch_step_stream(const StepArgs& a, size_t smem, int grid, int threads,
                               cudaStream_t st) {
  // The fold units' update on the tensor cores when REPLAYSSM_FOLD_TENSOR_CORES
  // is set to 1 (a measured alternative, slower here: see the header).
  const char* tc = std::getenv("REPLAYSSM_FOLD_TENSOR_CORES");
  auto kern = tc && tc[0] == '1' ? mamba2_step_stream_kernel<N, TS, TV, true>
                                 : mamba2_step_stream_kernel<N, TS, TV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // a programmatic dependent of the coefficient kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

cudaError_t launch_mamba2_fold_decode(const replayssm_dims& d, const replayssm_state& s,
                                      const float* A, const float* D, const void* x,
                                      const void* B, const void* C, const float* dt, float* y,
                                      cudaStream_t st) {
  const bool rd16 = s.S_read != nullptr, in16 = d.in_dtype == REPLAYSSM_BF16;
  const int ts = rd16 ? 2 : 4, FS = 4 / ts;
  // the plain decode's tile: about 16 KB of state rows per unit
  int RB = std::max(32, (int)(16384 / (d.dk * ts)) / 32 * 32);
  RB = std::min(RB, d.dv);
  while (d.dv % RB) RB -= 32;
  const int GU = RB % 64 == 0 ? 2 : 1;
  const DeviceInfo& dev = device_info();
  const int nrb = d.dv / RB;
  const long long units = (long long)d.batch * d.heads * nrb;
  if (units >= (1LL << 31)) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>(units, dev.sms);
  const int nloc_max = (int)((units + grid - 1) / grid);  // units of the largest block
  const int threads = 32 * (kStreamGroups * GU + 1);
  const int xblk = d.window * d.dv * (in16 ? 2 : 4);  // a head's ring x block
  const StepSmem fixed(RB, d.dk, ts, 0, nloc_max, xblk);
  const size_t per_stage = fixed.stage + fixed.side + 16;
  // stages: a multiple of the consumer groups (each owns NS / 4 of them),
  // at most 12, and each group's share holds a fold unit's FS stages
  const size_t room = (size_t)dev.smem_optin > fixed.total + 2048
                          ? ((size_t)dev.smem_optin - fixed.total - 2048) / per_stage : 0;
  const int NS = (int)std::min<size_t>(room, 12) / kStreamGroups * kStreamGroups;
  // Each consumer warp takes 32 rows of a unit, and a fold unit's FP32 rows
  // give each warp whole stages (or share one); the entries must fit the
  // registers. Otherwise: fold, then decode.
  if (d.window > kStepMaxW || RB / GU != 32 || (FS > 1 && GU != FS) ||
      NS < kStreamGroups * FS) {
    cudaError_t e = launch_mamba2_fold(d, s, A, 1, 0, st);
    if (e != cudaSuccess) return e;
    return launch_mamba2_decode(d, s, A, D, x, B, C, dt, y, st);
  }
  const size_t smem = StepSmem(RB, d.dk, ts, NS, nloc_max, xblk).total;

  const StepLayout sl(d);
  M2Coef p{d.batch, d.heads, d.groups, d.window, A, D, B, C, dt,
           s.ring_B, s.ring_C, s.ring_dt, s.ring_head, s.ring_len, s.status,
           s.work, s.work + sl.bf0};
  cudaError_t e = launch_step_coef(d, p, st);
  if (e != cudaSuccess) return e;

  StepArgs a{};
  a.batch = d.batch;
  a.H = d.heads;
  a.G = d.groups;
  a.P = d.dv;
  a.W = d.window;
  a.RB = RB;
  a.nrb = nrb;
  a.NS = NS;
  a.GU = GU;
  a.nloc_max = nloc_max;
  a.S = rd16 ? (const void*)s.S_read : (const void*)s.S_ckpt;
  a.S_ckpt = s.S_ckpt;
  a.S_read = reinterpret_cast<bf16*>(s.S_read);
  a.out = y;
  a.work = s.work;
  a.xblk = xblk;
  a.bfold = s.work + sl.bf0;
  a.x = x;
  a.C = C;
  a.ring_x = s.ring_x;
  a.head = s.ring_head;
  a.len = s.ring_len;
  a.status = s.status;
  a.sync = s.sync;
  if (d.dk == 128) {
    if (rd16) return in16 ? launch_step_stream<128, bf16, bf16>(a, smem, grid, threads, st)
                          : launch_step_stream<128, bf16, float>(a, smem, grid, threads, st);
    return in16 ? launch_step_stream<128, float, bf16>(a, smem, grid, threads, st)
                : launch_step_stream<128, float, float>(a, smem, grid, threads, st);
  }
  if (rd16) return in16 ? launch_step_stream<64, bf16, bf16>(a, smem, grid, threads, st)
                        : launch_step_stream<64, bf16, float>(a, smem, grid, threads, st);
  return in16 ? launch_step_stream<64, float, bf16>(a, smem, grid, threads, st)
              : launch_step_stream<64, float, float>(a, smem, grid, threads, st);
}

}  // namespace rs
