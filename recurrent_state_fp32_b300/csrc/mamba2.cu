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

constexpr int kM2MaxConsumers = 8;                         // consumer warps per block (4 or 8)
constexpr int kM2MaxThreads = 32 * (kM2MaxConsumers + 1);  // + one producer warp
constexpr int kRunHeads = 32;  // heads per run: producer lane h owns head h of the run
constexpr int kRunBufs = 3;    // run buffers (prefetch depth two runs)

struct M2Decode {
  int batch, H, G, P, W, NS, RB, nrb;  // RB state rows per stage, nrb = P / RB stages per head
  int GU;                              // consumer warps sharing a unit (1 or 2)
  const void* S;  // read copy (bf16) or checkpoint (f32)
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

// Scalars of one run (a stretch of units sharing a sequence and B/C group).
struct M2Run {
  int seq, h0, len, hd, ok, i_end;  // i_end: block-local index one past the run's last unit
};

// Shared-memory layout (byte offsets) of the persistent decode block.
// Stage: RB state rows, the head's buffered x rows (entry order), the index
// of the run buffer the unit belongs to. Run buffer: raw data (buffered B
// slots, C, B of the token, the run's current x and ring dt rows, dt/A/D,
// pointers) and what the producer derives once per run (C as floats, the
// per-head weights w_j (C.B_j) for every entry, decay, run scalars).
struct M2Layout {
  size_t tile, xr, sidx, stage;
  size_t rB, rC, rBt, rXt, rDt, rS, rCf, rCB, rCoef, rDecay, rMeta, run;
  size_t stages, runs, bars, total;
  __host__ __device__ M2Layout(int P, int N, int W, int RB, int ts, int ti, int NS) {
    const int Wd = ring_wd(W);
    tile = 0;
    xr = align_up((size_t)RB * N * ts, 128);
    sidx = xr + align_up((size_t)W * P * ti, 16);
    stage = align_up(sidx + 16, 128);
    rB = 0;
    rC = rB + align_up((size_t)W * N * ti, 16);
    rBt = rC + align_up((size_t)N * ti, 16);
    rXt = rBt + align_up((size_t)N * ti, 16);
    rDt = rXt + (size_t)kRunHeads * P * ti;
    rS = rDt + (size_t)kRunHeads * Wd * 4;                 // dt, A, D per head, then len, head
    rCf = rS + align_up((3 * (size_t)kRunHeads + 4) * 4, 16);
    rCB = rCf + (size_t)N * 4;                             // C.B per entry (W + 1 with the token)
    rCoef = rCB + align_up((size_t)(W + 1) * 4, 16);       // [kRunHeads][W + 1]
    rDecay = rCoef + align_up((size_t)kRunHeads * (W + 1) * 4, 16);
    rMeta = rDecay + (size_t)kRunHeads * 4;
    run = align_up(rMeta + sizeof(M2Run), 128);
    stages = 0;
    runs = stages + (size_t)NS * stage;
    bars = runs + kRunBufs * run;
    total = bars + (2 * (size_t)NS + 2 * kRunBufs) * 8;
  }
};

// Persistent replay decode.
//
// Work is split in units (sequence, head, row block of RB state rows); block
// b owns the units with flat index in [u0, u1) (a balanced split). The last
// warp is the producer, the others are consumers.
//
// The producer walks the range in runs of at most 32 heads that share a
// sequence and a B/C group. Two runs ahead it prefetches a run's raw data
// into a run buffer (bulk copies and 4-byte async copies). At a run's start
// it derives, once, C as floats, C.B_j of every buffered entry (a
// reduce-scatter over 16 entries at a time) and, lane h for head h, the
// weights w_j (C.B_j) and the decay by a serial suffix sum over the entries.
// Per unit it only issues the unit's bulk copies (state rows; the head's
// buffered x rows, one or two pieces), one instruction across three lanes.
//
// Consumer c takes the block's units i = c, c + C, ... (stage i mod NS; NS
// is a multiple of C, so a stage always has the same consumer and parity
// waits cannot alias): buffer terms of its rows from the run's weights, the
// rows through the row-dot engine, the output; the unit with row block 0
// appends the head's x and dt to the ring. After its last unit of a run a
// consumer arrives on the run buffer's "consumed" barrier, which the
// producer waits on before reusing the buffer. The block arrives on the
// sequences it covered at the end; the last arrival bumps len.
template <int N, typename TS, typename TI>
__global__ void __launch_bounds__(kM2MaxThreads, 1) mamba2_decode_kernel(const M2Decode a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using RD = RowDot<N, TS>;
  // A warp's 32 rows fit in 64 registers per lane: copy them out and free the stage early.
  constexpr bool kEarlyRelease = RD::kLpr <= 16;
  constexpr int kNL = N / 32;  // C elements per producer lane
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CW = (int)(blockDim.x / 32) - 1;  // consumer warps; the producer is warp CW
  const int GU = a.GU, NG = CW / GU;          // warps per unit, consumer groups
  const int H = a.H, G = a.G, P = a.P, W = a.W, NS = a.NS, hpg = H / G, nrb = a.nrb;
  const int RB = a.RB, Wd = ring_wd(W), W1 = W + 1;
  const M2Layout L(P, N, W, RB, sizeof(TS), sizeof(TI), NS);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + NS;
  uint64_t* rbar = empty + NS;          // run data landed
  uint64_t* consumed = rbar + kRunBufs;  // run buffer free again
  __shared__ int abort_smem;
  volatile int& abort_flag = abort_smem;
  const long long per_seq = (long long)H * nrb;
  const long long units = (long long)a.batch * per_seq;
  const long long u0 = units * blockIdx.x / gridDim.x;
  const long long u1 = units * (blockIdx.x + 1) / gridDim.x;
  const int my_units = (int)(u1 - u0);
  const TI* Bin = reinterpret_cast<const TI*>(a.B);
  const TI* Cin = reinterpret_cast<const TI*>(a.C);
  const TI* xin = reinterpret_cast<const TI*>(a.x);
  const TS* Sg = reinterpret_cast<const TS*>(a.S);
  const uint32_t tile_bytes = (uint32_t)((size_t)RB * N * sizeof(TS));
  const uint32_t row = (uint32_t)(P * sizeof(TI));  // bytes of one x row
  auto stage_ptr = [&](int s) { return smem + L.stages + (size_t)s * L.stage; };
  auto run_ptr = [&](int r) { return smem + L.runs + (size_t)r * L.run; };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], GU);
    }
    for (int r = 0; r < kRunBufs; ++r) {
      mbar_init(&rbar[r], 1);
      mbar_init(&consumed[r], CW);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();

  if (warp == CW) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_evict_first_policy();
    // End (exclusive unit index) of the run starting at unit u: same
    // sequence and group, at most kRunHeads heads.
    auto run_end = [&](long long u) {
      const long long seq = u / per_seq;
      const int h = (int)((u - seq * per_seq) / nrb);
      const int g_end = (h / hpg + 1) * hpg;
      const int h_end = min(g_end, h + kRunHeads);
      return min(u1, (seq * H + h_end) * nrb);
    };
    // Issue the copies of run [u, e) into run buffer r.
    auto prefetch = [&](long long u, long long e, int r) {
      const int seq = (int)(u / per_seq);
      const int h0 = (int)((u - (long long)seq * per_seq) / nrb), g = h0 / hpg;
      const int nh = (int)((e - 1 - (long long)seq * per_seq) / nrb) - h0 + 1;
      unsigned char* rb = run_ptr(r);
      float* rs = reinterpret_cast<float*>(rb + L.rS);
      if (lane < nh) {
        cp_async4(rs + lane, a.dt + (size_t)seq * H + h0 + lane);
        cp_async4(rs + kRunHeads + lane, a.A + h0 + lane);
        cp_async4(rs + 2 * kRunHeads + lane, a.D + h0 + lane);
      }
      if (lane == 0) {
        cp_async4(rs + 3 * kRunHeads, a.len + seq);
        cp_async4(rs + 3 * kRunHeads + 1, a.head + seq);
      }
      cp_async_commit();  // one group per run
      if (lane == 0) {
        const uint32_t nb = (uint32_t)(N * sizeof(TI));
        mbar_arrive_expect_tx(&rbar[r], nb * (W + 2) + (uint32_t)nh * (row + Wd * 4));
        const TI* rBsrc = reinterpret_cast<const TI*>(a.ring_B) + ((size_t)seq * W * G + g) * N;
        if (G == 1) {
          bulk_g2s(rb + L.rB, rBsrc, nb * W, &rbar[r]);
        } else {
          for (int w = 0; w < W; ++w)
            bulk_g2s(rb + L.rB + (size_t)w * nb, rBsrc + (size_t)w * G * N, nb, &rbar[r]);
        }
        bulk_g2s(rb + L.rC, Cin + ((size_t)seq * G + g) * N, nb, &rbar[r]);
        bulk_g2s(rb + L.rBt, Bin + ((size_t)seq * G + g) * N, nb, &rbar[r]);
        bulk_g2s(rb + L.rXt, xin + ((size_t)seq * H + h0) * P, (uint32_t)nh * row, &rbar[r]);
        bulk_g2s(rb + L.rDt, a.ring_dt + ((size_t)seq * H + h0) * Wd, (uint32_t)nh * Wd * 4,
                 &rbar[r]);
      }
    };
    // Runs k = 0, 1, ... use buffer k mod 3; phases count uses per buffer.
    uint32_t rphase = 0, cphase = 0;  // bit r: parity of rbar[r] / consumed[r] to wait for
    long long u = u0;
    long long e = u < u1 ? run_end(u) : u1;          // end of run k
    long long e1 = e < u1 ? run_end(e) : u1;         // end of run k + 1
    if (u < u1) prefetch(u, e, 0);
    if (e < u1) prefetch(e, e1, 1);
    int k = 0, r = 0;
    int ps = 0;          // stage of the next unit
    uint32_t pk = 0;     // parity of the empty-barrier phase to wait for on stage ps
    bool pwrap = false;  // stages are being reused (the first NS units need no wait)
    bool stop = false;   // warp-uniform
    int i = 0;           // block-local unit index
    while (u < u1 && !stop && !__shfl_sync(kFull, abort_flag, 0)) {
      // ---- run start: wait for its data, derive the run's values
      if (e < u1)
        cp_async_wait_group<1>();  // the next run's group may still be in flight
      else
        cp_async_wait_group<0>();
      const bool run_ok = mbar_wait_warp(&rbar[r], (rphase >> r) & 1);
      rphase ^= 1u << r;
      __syncwarp();
      unsigned char* rb = run_ptr(r);
      const float* rs = reinterpret_cast<const float*>(rb + L.rS);
      const int seq = (int)(u / per_seq);
      const int h0 = (int)((u - (long long)seq * per_seq) / nrb), g = h0 / hpg;
      const int nh = (int)((e - 1 - (long long)seq * per_seq) / nrb) - h0 + 1;
      const int n_units = (int)(e - u);
      if (!run_ok) {
        if (lane == 0) {
          atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
          abort_flag = 1;
        }
        break;
      }
      const int len = reinterpret_cast<const int*>(rs)[3 * kRunHeads];
      const int hd = reinterpret_cast<const int*>(rs)[3 * kRunHeads + 1];
      const bool ok = pointers_ok(hd, len, W) && len + 1 <= W;
      if (!ok && u == (long long)seq * per_seq && lane == 0)
        atomicOr(a.status + seq, pointers_ok(hd, len, W) ? REPLAYSSM_SEQ_RING_FULL
                                                         : REPLAYSSM_SEQ_BAD_POINTER);
      if (ok) {
        const TI* Cr = reinterpret_cast<const TI*>(rb + L.rC);
        const TI* Br = reinterpret_cast<const TI*>(rb + L.rB);
        const TI* Btr = reinterpret_cast<const TI*>(rb + L.rBt);
        float* Cf = reinterpret_cast<float*>(rb + L.rCf);
        float* CB = reinterpret_cast<float*>(rb + L.rCB);
        float cf[kNL];
#pragma unroll
        for (int q = 0; q < kNL; ++q) {
          cf[q] = to_f(Cr[lane + 32 * q]);
          Cf[lane + 32 * q] = cf[q];
        }
        // C.B_j for entries j < len, 16 at a time: lanes l and l + 16 end up
        // with entry j0 + (l mod 16).
        for (int j0 = 0; j0 < len; j0 += 16) {
          float v[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int j = j0 + t;
            const int slot = (hd + min(j, len - 1)) % W;
            float p = 0.f;
#pragma unroll
            for (int q = 0; q < kNL; ++q) p = fmaf(cf[q], to_f(Br[(size_t)slot * N + lane + 32 * q]), p);
            v[t] = p;
          }
          float tot = reduce_scatter<16>(v, lane);
          tot += __shfl_xor_sync(kFull, tot, 16);
          const int j = j0 + (lane & 15);
          if (lane < 16 && j < len) CB[j] = tot;
        }
        float cbt = 0.f;
#pragma unroll
        for (int q = 0; q < kNL; ++q) cbt = fmaf(cf[q], to_f(Btr[lane + 32 * q]), cbt);
        cbt = warp_sum(cbt);
        if (lane == 0) CB[len] = cbt;
        __syncwarp();
        // lane h: weights of head h0 + h, newest entry first
        if (lane < nh) {
          const float Ah = rs[kRunHeads + lane];
          const float* dtr = reinterpret_cast<const float*>(rb + L.rDt) + (size_t)lane * Wd;
          float* coef = reinterpret_cast<float*>(rb + L.rCoef) + (size_t)lane * W1;
          float acc = rs[lane];  // dt of the token (entry len)
          coef[len] = acc * CB[len];
          for (int j = len - 1; j >= 0; --j) {
            const float dtj = dtr[(hd + j) % W];
            coef[j] = dtj * expf(Ah * acc) * CB[j];
            acc += dtj;
          }
          reinterpret_cast<float*>(rb + L.rDecay)[lane] = expf(Ah * acc);
        }
        // Ring append of the group's B and C, once per (sequence, group): by the
        // run that starts at the group's first unit.
        if (h0 % hpg == 0 && u == ((long long)seq * H + h0) * nrb) {
          const int slot = (hd + len) % W;
          TI* dB = reinterpret_cast<TI*>(a.ring_B) + (((size_t)seq * W + slot) * G + g) * N;
          for (int c = lane; c < N; c += 32) dB[c] = Btr[c];
          if (a.ring_C) {
            TI* dC = reinterpret_cast<TI*>(a.ring_C) + (((size_t)seq * W + slot) * G + g) * N;
            for (int c = lane; c < N; c += 32) dC[c] = Cr[c];
          }
        }
      }
      if (lane == 0) {
        M2Run* m = reinterpret_cast<M2Run*>(rb + L.rMeta);
        m->seq = seq;
        m->h0 = h0;
        m->len = len;
        m->hd = hd;
        m->ok = ok;
        m->i_end = i + n_units;
        // consumers with no unit in this run arrive now on their behalf
        const int absent = CW - GU * min(NG, n_units);
        if (absent > 0) mbar_arrive_cnt(&consumed[r], (uint32_t)absent);
      }
      __syncwarp();

      // ---- units of this run
      int hu = h0, rbk = (int)(u - ((long long)seq * H + h0) * nrb);  // head, row block
      for (; u < e; ++u, ++i) {
        const int s = ps;
        if (pwrap && !mbar_wait_warp(&empty[s], pk)) {
          if (lane == 0) abort_flag = 1;
          stop = true;
          break;
        }
        if (++ps == NS) {  // the next unit reuses stage 0: wait for one more phase
          ps = 0;
          if (pwrap) pk ^= 1;
          pwrap = true;
        }
        unsigned char* st = stage_ptr(s);
        if (lane == 0) {
          *reinterpret_cast<int*>(st + L.sidx) = r;
          if (ok) {
            // one bulk copy per unit: the unit's state rows (about 16 KB)
            mbar_arrive_expect_tx(&full[s], tile_bytes);
            bulk_g2s(st + L.tile, Sg + (((size_t)seq * H + hu) * P + (size_t)rbk * RB) * N,
                     tile_bytes, &full[s], pol);
          } else {
            mbar_arrive(&full[s]);  // the consumer skips the unit
          }
        }
        if (++rbk == nrb) {
          rbk = 0;
          ++hu;
        }
      }
      if (stop) break;
      // ---- prefetch run k + 2 into the buffer of run k - 1, once it is consumed
      const long long e2 = e1 < u1 ? run_end(e1) : u1;
      if (e1 < u1) {
        const int r2 = (r + 2) % kRunBufs;
        if (k >= 1 && !mbar_wait_warp(&consumed[r2], (cphase >> r2) & 1)) {
          if (lane == 0) abort_flag = 1;
          break;
        }
        if (k >= 1) cphase ^= 1u << r2;
        prefetch(e1, e2, r2);
      }
      e = e1;  // every run holds at least one unit, so the walk always advances
      e1 = e2;
      ++k;
      r = (r + 1) % kRunBufs;
    }
    cp_async_wait_all();
  } else {
    // ------------------------------------------------------------ consumers
    const int cpr = (int)(row / 16);  // 16-byte chunks per x row
    const int gi = warp / GU, part = warp - gi * GU;  // consumer group, part within it
    const int gt = part * 32 + lane;                  // thread index within the group
    // Syncs the GU warps of this group (named barrier 1 + gi).
    auto group_sync = [&]() {
      if (GU == 1)
        __syncwarp();
      else
        asm volatile("bar.sync %0, %1;" ::"r"(1 + gi), "r"(32 * GU) : "memory");
    };
    // Group sync that also ORs a (warp-uniform) flag over the group, so that
    // both warps of a group always take the same exit decision.
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
    // Async copies (this thread's share) of the buffered x rows of global
    // head hg (entries 0..len-1, oldest first) into dst; one commit group.
    auto fetch_xrows = [&](unsigned char* dst, int hg, int len, int hd) {
      const unsigned char* base = reinterpret_cast<const unsigned char*>(a.ring_x) +
                                  (size_t)hg * W * row;
      for (int idx = gt; idx < len * cpr; idx += 32 * GU) {
        const int j = idx / cpr, c = idx - j * cpr;
        cp_async16(dst + (size_t)j * row + c * 16, base + (size_t)((hd + j) % W) * row + c * 16);
      }
      cp_async_commit();
    };
    int s = gi;       // stage of this group's next unit (NS is a multiple of NG)
    uint32_t ph = 0;  // its full-barrier phase parity
    bool pre = false;  // the x rows of this group's next unit are already requested
    const int RBp = RB / GU;  // rows of a unit handled by this warp
    for (int i = gi; i < my_units; i += NG) {
      const bool aborted = __shfl_sync(kFull, abort_flag, 0) != 0;
      const bool landed = !aborted && mbar_wait_warp(&full[s], ph);
      if (!aborted && !landed && lane == 0) {
        abort_flag = 1;
        atomicOr(a.status + (int)((u0 + i) / per_seq), REPLAYSSM_SEQ_TIMEOUT);
      }
      // one decision per group; also: the group's other warp is done with its
      // previous unit
      if (group_any(!landed)) break;
      unsigned char* st = stage_ptr(s);
      const int r = *reinterpret_cast<const int*>(st + L.sidx);
      const unsigned char* rb = run_ptr(r);
      const M2Run m = *reinterpret_cast<const M2Run*>(rb + L.rMeta);
      bool released = false;  // this warp already freed the stage's state rows
      const int u = (int)(u0 + i);  // unit counts fit in 32 bits (checked on the host)
      const int hg = u / nrb;       // global head index seq * H + h
      const int rbk = u - hg * nrb;
      // next unit of this group: stage s2; prefetch its x rows if it is in this run
      int s2 = s + NG, ph2 = ph;
      if (s2 >= NS) {
        s2 -= NS;
        ph2 ^= 1;
      }
      if (m.ok) {
        if (!pre) fetch_xrows(st + L.xr, hg, m.len, m.hd);
        // (needs a second stage per group: NS >= 2 NG)
        const bool next_here = NS >= 2 * NG && i + NG < m.i_end;
        if (next_here) {
          const int hg2 = (u + NG) / nrb;
          fetch_xrows(stage_ptr(s2) + L.xr, hg2, m.len, m.hd);
          cp_async_wait_group<1>();  // this unit's rows have landed
        } else {
          cp_async_wait_group<0>();
        }
        pre = next_here;
        group_sync();  // every thread's share of the rows is visible
        const int len = m.len, hd = m.hd;
        const int h = hg - m.seq * H, hi = h - m.h0;
        const float* rs = reinterpret_cast<const float*>(rb + L.rS);
        const float* coef = reinterpret_cast<const float*>(rb + L.rCoef) + (size_t)hi * W1;
        const float decay = reinterpret_cast<const float*>(rb + L.rDecay)[hi];
        const TI* xt = reinterpret_cast<const TI*>(rb + L.rXt) + (size_t)hi * P;
        const TI* xr = reinterpret_cast<const TI*>(st + L.xr);
        // buffer terms of this unit's rows: extra[p] = sum_j coef_j x_j[p] + D x[p]
        const float c_tok = rs[2 * kRunHeads + hi] + coef[len];
        const int pbase = rbk * RB + part * RBp;
        float ex[2] = {0.f, 0.f};  // rows pbase + 2 lane + {0, 1} (+64 for the second pair)
        float ex2[2] = {0.f, 0.f};
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const int q = 2 * lane + 64 * pp;
          if (q < RBp) {
            float2 xv = load2<TI>(xt + pbase + q);
            float e0 = c_tok * xv.x, e1 = c_tok * xv.y;
#pragma unroll 4
            for (int j = 0; j < len; ++j) {
              const float c = coef[j];
              xv = load2<TI>(xr + (size_t)j * P + pbase + q);
              e0 = fmaf(c, xv.x, e0);
              e1 = fmaf(c, xv.y, e1);
            }
            if (pp == 0) {
              ex[0] = e0;
              ex[1] = e1;
            } else {
              ex2[0] = e0;
              ex2[1] = e1;
            }
          }
        }
        // ring append of this head's x and dt (once per head: row block 0)
        if (rbk == 0 && part == 0) {
          const int slot = (hd + len) % W;
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(a.ring_x) +
                                                ((size_t)hg * W + slot) * row);
          const uint4* src = reinterpret_cast<const uint4*>(xt);
          for (int c = lane; c < cpr; c += 32) dst[c] = src[c];
          if (lane == 0) a.ring_dt[(size_t)hg * Wd + slot] = rs[hi];
        }
        float vec[RD::kEpc];
        const float* cv = reinterpret_cast<const float*>(rb + L.rCf) + RD::chunk_of(lane) * RD::kEpc;
#pragma unroll
        for (int e2 = 0; e2 < RD::kEpc; ++e2) vec[e2] = cv[e2];
        const TS* tile = reinterpret_cast<const TS*>(st + L.tile) + (size_t)part * RBp * N;
        float* yrow = a.y + (size_t)hg * P + pbase;
        // row r of the unit lives in lane (r / 2) mod 32 (pair r mod 2, set r / 64)
        auto extra_of = [&](int rr) {
          const int src_lane = (rr >> 1) & 31;
          const float e0 = __shfl_sync(kFull, (rr & 64) ? ex2[0] : ex[0], src_lane);
          const float e1 = __shfl_sync(kFull, (rr & 64) ? ex2[1] : ex[1], src_lane);
          return (rr & 1) ? e1 : e0;
        };
        int row0 = 0;
        if (kEarlyRelease && RBp == 32) {
          // copy this warp's 32 rows to registers and free the stage at once,
          // so the next copy into it starts while the arithmetic runs
          uint4 raw[RD::kLpr];
          RD::load32(tile, 0, lane, raw);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          released = true;
          const float dot = RD::dot32(raw, vec, lane);
          const int rr = RD::row_of(lane);
          const float xa = extra_of(rr);
          yrow[rr] = fmaf(decay, dot, xa);
          row0 = RBp;
        }
        for (; row0 + 64 <= RBp; row0 += 64) {
          float d0, d1;
          RD::rows32x2(tile, row0, row0 + 32, vec, lane, d0, d1);
          const int ra = row0 + RD::row_of(lane), rb2 = ra + 32;
          const float xa = extra_of(ra), xb = extra_of(rb2);
          yrow[ra] = fmaf(decay, d0, xa);
          yrow[rb2] = fmaf(decay, d1, xb);
        }
        if (row0 < RBp) {
          const float dot = RD::rows32(tile, row0, vec, lane);
          const int rr = row0 + RD::row_of(lane);
          const float xa = extra_of(rr);
          yrow[rr] = fmaf(decay, dot, xa);
        }
      } else {
        pre = false;
      }
      __syncwarp();
      if (lane == 0) {
        if (!released) mbar_arrive(&empty[s]);
        if (i + NG >= m.i_end) mbar_arrive(&consumed[r]);  // last unit of this run here
      }
      s = s2;
      ph = ph2;
    }
    cp_async_wait_all();
  }
  __syncthreads();
  // No bulk copy may land after the block exits.
  if (tid == 0 && abort_flag) {
    for (int s = 0; s < NS + kRunBufs; ++s) {  // the NS stages and the run buffers
      uint64_t* b = s < NS ? &full[s] : &rbar[s - NS];
      mbar_wait(b, 0);
      mbar_wait(b, 1);
    }
  }
  // Arrive on every sequence this block covered; the last block bumps len.
  if (u0 < u1) {
    const int s0 = (int)(u0 / per_seq), s1 = (int)((u1 - 1) / per_seq);
    for (int seq = s0 + tid; seq <= s1; seq += blockDim.x) {
      const int len = a.len[seq], hd = a.head[seq];
      if (!pointers_ok(hd, len, W) || len + 1 > W) continue;
      const long long a0 = max(u0, (long long)seq * per_seq);
      const long long a1 = min(u1, (long long)(seq + 1) * per_seq);
      arrive_and_finish(a.sync + seq, (int)(a1 - a0), (int)per_seq,
                        [&] { a.len[seq] = len + 1; });
    }
  }
}

template <int N, typename TS, typename TI>
cudaError_t decode_inst(M2Decode a, cudaStream_t st) {
  const DeviceInfo& dev = device_info();
  // One bulk copy of about 16 KB of state rows per unit: smaller copies
  // are dominated by the fixed cost of a bulk copy.
  int RB = std::max(32, (int)(16384 / (N * sizeof(TS))) / 32 * 32);
  RB = std::min(RB, a.P);
  while (a.P % RB) RB -= 32;
  a.RB = RB;
  a.nrb = a.P / RB;
  const M2Layout one(a.P, N, a.W, RB, sizeof(TS), sizeof(TI), 1);
  const size_t fixed = one.total - one.stage - 2 * 8;
  const int fit = (int)(((size_t)dev.smem_optin - fixed - 1024) / (one.stage + 16));
  // Four consumer groups; NS a multiple of 4 (two stages per group when
  // they fit): a stage always has the same group, so parity waits cannot
  // alias, and a group fetches its next unit's x rows into its other stage.
  // Units of 64, 128, ... rows are shared by two warps (each half the rows).
  const int NG = 4;
  a.GU = RB % 64 == 0 ? 2 : 1;  // each warp's share must be whole 32-row groups
  const int C = NG * a.GU;
  const int NS = std::min(fit, 2 * NG) / NG * NG;
  if (NS < NG) return cudaErrorInvalidConfiguration;
  a.NS = NS;
  const M2Layout L(a.P, N, a.W, RB, sizeof(TS), sizeof(TI), NS);
  auto kern = mamba2_decode_kernel<N, TS, TI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L.total);
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.batch * a.H * a.nrb;
  if (units >= (1LL << 31)) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>(units, dev.sms);
  kern<<<grid, 32 * (C + 1), L.total, st>>>(a);
  return cudaGetLastError();
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
        const float dtj = a.ring_dt[((size_t)seq * H + h) * ring_wd(W) + (hd + j) % W];
        s_w[j] = dtj * expf(Ah * acc);
        acc += dtj;
      }
      s_decay = expf(Ah * acc);
    }
    __syncthreads();
    for (int idx = tid; idx < n * P; idx += kThreads) {
      const int j = idx / P, p = idx - j * P;
      xw[idx] = s_w[j] * to_f(rx[(((size_t)seq * H + h) * W + (hd + j) % W) * P + p]);
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

}  // namespace

cudaError_t launch_mamba2_decode(const replayssm_dims& d, const replayssm_state& s, const float* A,
                                 const float* D, const void* x, const void* B, const void* C,
                                 const float* dt, float* y, cudaStream_t st) {
  const bool rd16 = s.S_read != nullptr;
  M2Decode a{d.batch, d.heads, d.groups, d.dv, d.window, 0, 0, 0, 1,
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
