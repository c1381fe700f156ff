// Stream kernel of the fused Mamba-2 fold + decode step.
//
// One decode step that also performs the consolidation it needs: a
// sequence whose ring is full is folded before its token is decoded, and the
// fold happens while its state rows stream past, so the FP32 checkpoint is
// read once, written once (with its BF16 read copy) and its output comes
// from the new rows. The checkpoint-plus-ring split and "fold only when the
// buffer fills" follow "NVIDIA y Princeton aceleran modelos híbridos al
// guardar entradas recientes en lugar del estado completo", paragraph 2.
//
// A short coefficient grid runs first (mamba2_step_coef_kernel): per head
// the decode weights c_j = w_j (C . B_j) of the l buffered entries, the
// token's weight c_tok (with D), the decode decay, and for a fold the fold
// weights and fold decay. This kernel is its programmatic dependent: its
// producer streams state rows at once, its consumers wait for the weights.
//
// Units are (sequence, head, row block of RB rows), dealt to the blocks in
// turn (unit u goes to block u mod grid), so the folds of any set of
// sequences spread over all SMs. In each block a producer warp fills a ring
// of NS shared-memory stages with one bulk copy per stage and consumer
// groups of GU warps take the block's units round robin. Two kinds of unit:
//   decode  (ring not full): one stage of read-copy rows;
//           y[r] = decay * (S[r, :] . C) + sum_{j<l} c_j x_j[r] + c_tok x[r]
//           with the ring x rows x_j loaded by the consumer itself
//   fold    (ring full, n = len entries): FS = 4 / sizeof(TS) stages of FP32
//           checkpoint rows, the head's ring x block beside the first;
//           c_j[r] = w_j x_j[r],
//           S'[r, :] = fold_decay * S[r, :] + sum_j c_j[r] B_j,
//           S' written to the checkpoint and read copy, then
//           y[r] = decay * (S'_read[r, :] . C) + c_tok x[r]
// where S'_read is the row as the read copy holds it (the BF16 rounding when
// there is one), so outputs equal those of a consolidate then a decode. Each
// unit then appends the token's x for its own rows (with a fold, into entry
// 0's slot: no unit reads another unit's rows, and a fold unit's own rows
// were copied before it writes).
// The kind of every unit is fixed at block start from the ring pointers,
// which nothing changes until the last unit of a sequence is done: each
// block arrives on a sequence's counter once per unit of it when all its
// units are done, and the last arrival moves the pointers (fold:
// head += len, len = 1; else len += 1).
//
// Each consumer group owns R = NS / 4 of the stages and uses them in turn
// for its units (a fold unit takes FS consecutive ones), so a group only
// waits for a stage's next fill after it has consumed the previous one and
// the mbarrier parity of a wait cannot alias an older phase. The producer
// fills the stages of unit i's group in unit order.
#pragma once

#include "common.cuh"
#include "launch.h"
#include "stream.cuh"

namespace rs {

struct StepArgs {
  int batch, H, G, P, W, RB, nrb, NS, GU, nloc_max, xblk;
  const void* S;        // decode rows: the read copy, or the checkpoint without one
  float* S_ckpt;        // FP32 checkpoint [b, H, P, N]
  bf16* S_read;         // BF16 read copy or null
  float* out;           // y [b, H, P]
  const float* work;    // rows of kStepRow floats per (sequence, head), StepLayout
  const float* bfold;   // folded B rows [b, G, kStepMaxW, N]
  const void* x;        // token input x [b, H, P]
  const void* C;        // token input C [b, G, N]
  void* ring_x;         // [b, H, W, P]
  int32_t* head;
  int32_t* len;
  int32_t* status;
  int32_t* sync;
};

// Shared memory: NS stages, NS side buffers, full and empty barriers, and
// the entry of each of the block's units. A fold unit's first side buffer
// receives the head's ring x block (W x P inputs); then the side buffer of
// each of its stages holds the fold coefficients of that stage's FP32 rows.
struct StepSmem {
  size_t stage, side, sides, bars, table, total;
  __host__ __device__ StepSmem(int RB, int N, int ts, int NS, int nloc_max, int xblk) {
    stage = stream_stage_bytes(RB, N, ts);
    const size_t coefs = (size_t)(RB / (4 / ts)) * kStepMaxW * 4;  // a stage's rows
    side = align_up((size_t)xblk > coefs ? (size_t)xblk : coefs, 16);
    sides = (size_t)NS * stage;
    bars = sides + (size_t)NS * side;
    table = bars + 2 * (size_t)NS * 8;
    total = table + (size_t)nloc_max * 4;
  }
};

// Partial sums of CS rows spread over groups of L lanes (one chunk of each
// row per lane): log2(CS) reduce-scatter levels leave in each lane the row
// of the chunk given by its bits L/2, L/4, ... (most significant first),
// summed over those bits; xor shuffles sum the remaining low bits.
template <int L, int CS>
__device__ __forceinline__ float reduce_chunk(float (&v)[CS], int lane) {
#pragma unroll
  for (int o = L / 2, n = CS / 2; n >= 1; o >>= 1, n >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < n; ++k) {
      const float send = upper ? v[k] : v[k + n];
      const float keep = upper ? v[k + n] : v[k];
      v[k] = keep + __shfl_xor_sync(kFull, send, o);
    }
  }
#pragma unroll
  for (int o = L / (2 * CS); o >= 1; o >>= 1) v[0] += __shfl_xor_sync(kFull, v[0], o);
  return v[0];
}

// Row (of 32) whose total lane `lane` keeps when chunk m goes to the lanes
// with (lane mod L / CS) == m: its row group lane / L, its chunk, and the row
// of the chunk from reduce_chunk.
template <int L, int RPI, int CS>
__device__ __forceinline__ int fold_row(int lane) {
  constexpr int M = L / CS;  // chunks
  int in_chunk = 0;
#pragma unroll
  for (int o = L / 2; o > L / (2 * CS); o >>= 1) in_chunk = 2 * in_chunk + ((lane & o) != 0);
  return lane / L + RPI * (CS * (lane & (M - 1)) + in_chunk);
}

// x as hi + lo, each a TF32 value (round to nearest): hi carries the top 11
// mantissa bits, lo most of the rest, so products of the pairs lose little
// against FP32.
__device__ __forceinline__ void tf32_split(float x, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(x - __uint_as_float(hi)));
}

// d += a b for one 16 x 8 x 8 TF32 tile (warp-wide): a in the row-major A
// fragment order, b in the column-major B order, d the accumulator fragment.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// MMA: the fold units' rank-n update on the tensor cores (mma.sync, TF32
// split in two) instead of FP32 FMAs; both give the same results within
// FP32 rounding.
template <int N, typename TS, typename TV, bool MMA>
__global__ void __launch_bounds__(kStreamMaxThreads, 1) mamba2_step_stream_kernel(const StepArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using RD = RowDot<N, TS>;     // decode units
  using RF = RowDot<N, float>;  // fold units (FP32 rows)
  constexpr int kE = RD::kEpc;
  constexpr bool kEarly = RD::kLpr <= 16;
  constexpr int FS = 4 / (int)sizeof(TS);      // stages per fold unit
  constexpr int kCS = 4;                       // rows per reduction chunk
  constexpr int kFoldChunks = RF::kLpr / kCS;  // chunks per lane and 32 rows
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CW = (int)(blockDim.x / 32) - 1;  // consumer warps; the producer is warp CW
  const int GU = a.GU, NG = CW / GU, NS = a.NS, H = a.H, P = a.P, RB = a.RB, nrb = a.nrb;
  const int W = a.W;
  const StepSmem L(RB, N, sizeof(TS), NS, a.nloc_max, a.xblk);
  const int R = NS / kStreamGroups;  // stages of each consumer group
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + NS;
  int* table = reinterpret_cast<int*>(smem + L.table);
  __shared__ int abort_smem;
  volatile int& abort_flag = abort_smem;
  const int per_seq = H * nrb;
  const long long units = (long long)a.batch * per_seq;
  const int G0 = (int)gridDim.x, b0 = (int)blockIdx.x;
  // local unit i is unit b0 + i * G0
  const int nloc = units > b0 ? (int)((units - b0 + G0 - 1) / G0) : 0;
  const uint32_t tile_bytes = (uint32_t)((size_t)RB * N * sizeof(TS));
  const uint32_t xblk = (uint32_t)a.xblk;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], GU);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  // Each local unit's entry: bit 0 pointers valid, bit 1 fold, len in bits
  // 8..15, head in bits 16..23.
  for (int i = tid; i < nloc; i += blockDim.x) {
    const int seq = (b0 + i * G0) / per_seq;
    const int l = a.len[seq], hd = a.head[seq];
    const bool ok = pointers_ok(hd, l, W);
    const bool fold = ok && l + 1 > W;
    table[i] = (ok ? 1 : 0) | (fold ? 2 : 0) | (ok ? (l << 8) | (hd << 16) : 0);
  }
  __syncthreads();

  if (warp == CW) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_evict_first_policy();
    const TS* Sg = reinterpret_cast<const TS*>(a.S);
    // Per consumer group (unit i belongs to group i mod 4): its next unit,
    // the stages of that unit already issued, its position in its R stages,
    // the parity of that fill and whether its stages are being refilled. The
    // groups are served in turn, each whenever its next stage is free, so a
    // group busy with a fold unit does not hold back the others.
    int nxt[kStreamGroups], fdone[kStreamGroups] = {}, t[kStreamGroups] = {};
    uint32_t ph[kStreamGroups] = {};
    bool reuse[kStreamGroups] = {};
#pragma unroll
    for (int gq = 0; gq < kStreamGroups; ++gq) nxt[gq] = gq;
    int left = nloc;     // units not yet fully issued
    uint64_t idle0 = 0;  // start of the current stretch without progress
    while (left > 0) {
      bool progress = false;
#pragma unroll
      for (int gq = 0; gq < kStreamGroups; ++gq) {
        const int i = nxt[gq];
        if (i >= nloc) continue;
        const int s = gq * R + t[gq];
        const bool room = !reuse[gq] || __shfl_sync(kFull, (int)mbar_try_wait(&empty[s], ph[gq] ^ 1), 0);
        if (!room) continue;
        const int u = b0 + i * G0;
        const int hg = nrb == 1 ? u : u / nrb, rb = u - hg * nrb;
        const bool fold = (table[i] & 2) != 0;
        const int f = fdone[gq];
        if (lane == 0) {
          const size_t row = (size_t)hg * P + (size_t)rb * RB;
          if (fold) {
            // FP32 rows; beside the first stage, the head's ring x block
            // (the token may or may not have reached entry 0's slot yet:
            // consumers take entry 0 from the saved row)
            const size_t r0 = row + (size_t)f * (RB / FS);
            mbar_arrive_expect_tx(&full[s], tile_bytes + (f == 0 ? xblk : 0));
            bulk_g2s(smem + (size_t)s * L.stage, a.S_ckpt + r0 * N, tile_bytes, &full[s], pol);
            if (f == 0)
              bulk_g2s(smem + L.sides + (size_t)s * L.side,
                       static_cast<const unsigned char*>(a.ring_x) + (size_t)hg * xblk, xblk,
                       &full[s]);
          } else {
            mbar_arrive_expect_tx(&full[s], tile_bytes);
            bulk_g2s(smem + (size_t)s * L.stage, Sg + row * N, tile_bytes, &full[s], pol);
          }
        }
        if (++t[gq] == R) {
          t[gq] = 0;
          ph[gq] ^= 1;
          reuse[gq] = true;
        }
        if (++fdone[gq] == (fold ? FS : 1)) {
          fdone[gq] = 0;
          nxt[gq] += kStreamGroups;
          --left;
        }
        progress = true;
      }
      if (progress) {
        idle0 = 0;
      } else {  // bounded: no stage freed for the wait limit ends the block's work
        const uint64_t now = global_ns();
        if (idle0 == 0) {
          idle0 = now;
        } else if (now - idle0 > kWaitLimitNs) {
          if (lane == 0) abort_flag = 1;
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int gi = warp / GU, part = warp - gi * GU;
    const int RBp = RB / GU;  // rows of a unit handled by this warp: 32 (launcher)
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
    const int cd = RD::chunk_of(lane) * kE;  // decode units: this lane's elements of C
    const int cf = RF::chunk_of(lane) * 4;   // fold units: this lane's four columns
    const TV* Cin = reinterpret_cast<const TV*>(a.C);
    const TV* xin = reinterpret_cast<const TV*>(a.x);
    TV* rx = reinterpret_cast<TV*>(a.ring_x);
    auto slot_of = [W](int s) { return s < W ? s : s - W; };
    // Work rows and folded B rows come from the preparation grid (this grid
    // may start before it ends).
    griddep_wait();
    int tg = 0;         // this group's position in its R stages
    uint32_t phg = 0;   // and the parity of that stage's fill
    for (int i = gi; i < nloc; i += NG) {
      const int u = b0 + i * G0;
      const int hg = nrb == 1 ? u : u / nrb, rb = u - hg * nrb;
      const int seq = hg / H, h = hg - seq * H;
      const int g = h / (H / a.G);
      const int code = table[i];
      const bool ok = (code & 1) != 0, fold = (code & 2) != 0;
      // the unit's stages in the group's ring: the first, and for a
      // two-stage fold unit the next one (wrapping flips the parity)
      const int s0 = gi * R + tg;
      const uint32_t ph0 = phg;
      const bool wrap1 = tg + 1 == R;
      const int s1 = gi * R + (wrap1 ? 0 : tg + 1);
      const uint32_t ph1 = wrap1 ? phg ^ 1 : phg;
      for (int f = 0; f < (fold ? FS : 1); ++f) {
        if (++tg == R) {
          tg = 0;
          phg ^= 1;
        }
      }
      const int row0 = rb * RB + part * RBp;  // first row of this warp within the head
      const float* w0 = a.work + (size_t)hg * kStepRow;
      float* yrow = a.out + (size_t)hg * P + row0;
      const float scale = w0[kStepDecay];
      const float ctok = w0[kStepTok];
      const int hd = (code >> 16) & 0xff, l = (code >> 8) & 0xff;
      // the token's ring slot: after the buffered entries, or entry 0's after a fold
      const int tslot = slot_of(fold ? hd : hd + l);
      const TV* xh = xin + (size_t)hg * P + row0;                 // the token's x rows
      TV* rxh = rx + (size_t)hg * W * P + row0;                   // the head's ring x rows
      const bool aborted = __shfl_sync(kFull, abort_flag, 0) != 0;
      if (!fold) {
        // -------------------------------------------------- decode unit
        // buffer terms of this lane's row from the ring x rows of the l
        // buffered entries, loaded before the wait for the state rows
        float vec[kE];
        load_vec<TV, kE>(Cin + ((size_t)seq * a.G + g) * N + cd, vec);
        const int r = RD::row_of(lane);
        const float cj = w0[lane & (kStepMaxW - 1)];
        const TV xtr = xh[r];
        TV xj[kStepMaxW];
#pragma unroll
        for (int j = 0; j < kStepMaxW; ++j)
          if (j < l) xj[j] = rxh[(size_t)slot_of(hd + j) * P + r];
        const int s = s0;
        const bool landed = !aborted && mbar_wait_warp(&full[s], ph0);
        if (!aborted && !landed && lane == 0) {
          abort_flag = 1;
          atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
        }
        if (group_any(!landed)) break;
        const TS* tile = reinterpret_cast<const TS*>(smem + (size_t)s * L.stage) + (size_t)part * RBp * N;
        float d;
        if constexpr (kEarly) {
          uint4 raw[RD::kLpr];
          RD::load32(tile, 0, lane, raw);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          d = RD::dot32(raw, vec, lane);
        } else {
          d = RD::rows32(tile, 0, vec, lane);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        float extra = ctok * to_f(xtr);
#pragma unroll
        for (int j = 0; j < kStepMaxW; ++j) {
          const float c = __shfl_sync(kFull, cj, j);
          if (j < l) extra = fmaf(c, to_f(xj[j]), extra);
        }
        if (ok) {
          yrow[r] = fmaf(scale, d, extra);
          rxh[(size_t)tslot * P + r] = xtr;  // append the token's x
        }
      } else {
        // ---------------------------------------------------- fold unit
        const int nf = l, hd0 = hd;
        const float fdec = w0[kStepFoldDecay];
        // B_j of the head's group, this lane's columns (zero past the n entries)
        const float* Bs = a.bfold + ((size_t)seq * a.G + g) * kStepMaxW * N + cf;
        float4 Bq[kStepMaxW];
        float c4[4];
        if constexpr (!MMA) {
#pragma unroll
          for (int j = 0; j < kStepMaxW; ++j)
            Bq[j] = j < nf ? *reinterpret_cast<const float4*>(Bs + (size_t)j * N)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
          load_vec<TV, 4>(Cin + ((size_t)seq * a.G + g) * N + cf, c4);
        }
        // the output row of this lane: one per lane, in the FMA loop's
        // reduction order or the tensor-core tiles' row order
        const int gq = lane >> 2, tq = lane & 3;
        const int r = MMA ? 16 * (tq >> 1) + gq + 8 * (tq & 1) : fold_row<RF::kLpr, RF::kRpi, kCS>(lane);
        const TV xtr = xh[r];  // the token (decoded after the fold, n = 1)
        const float extra = ctok * to_f(xtr);
        // this warp's stage: the unit's first, or the second of a two-stage
        // unit; the first also holds the ring x block, so every warp waits for it
        const bool second = FS > 1 && part == 1;
        const int s = second ? s1 : s0;
        bool landed = !aborted && mbar_wait_warp(&full[s0], ph0);
        if (second && landed) landed = mbar_wait_warp(&full[s1], ph1);
        if (!aborted && !landed && lane == 0) {
          abort_flag = 1;
          atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
        }
        if (group_any(!landed)) break;
        // coefficients c_j = w_j x_j of row row0 + lane from slot hd0 + j of
        // the copied ring x block: no warp writes this unit's rows of the
        // ring (the token goes into entry 0's slot) before the copy landed
        const int off = FS > 1 ? 0 : part * RBp;  // this warp's rows in its stage
        float* coef = reinterpret_cast<float*>(smem + L.sides + (size_t)s * L.side) +
                      (size_t)off * kStepMaxW;
        {
          const TV* xs = reinterpret_cast<const TV*>(smem + L.sides + (size_t)s0 * L.side);
          float cj[kStepMaxW];
#pragma unroll
          for (int j = 0; j < kStepMaxW; ++j)
            cj[j] = j < nf ? w0[kStepFoldW + j] * to_f(xs[(size_t)slot_of(hd0 + j) * P + row0 + lane]) : 0.f;
          // every warp of the unit has read the x block before any
          // coefficients overwrite it
          if (GU == 1) {
            __syncwarp();
          } else {
            asm volatile("bar.sync %0, %1;" ::"r"(1 + gi), "r"(32 * GU) : "memory");
          }
          float4* dst = reinterpret_cast<float4*>(coef + lane * kStepMaxW);
#pragma unroll
          for (int j = 0; j < kStepMaxW; j += 4) dst[j / 4] = make_float4(cj[j], cj[j + 1], cj[j + 2], cj[j + 3]);
          __syncwarp();
        }
        // this warp's 32 FP32 rows
        const float* tile = reinterpret_cast<const float*>(smem + (size_t)s * L.stage) + (size_t)off * N;
        float mine = 0.f;
        if constexpr (!MMA) {
        // rows in chunks of kCS per lane; lane l ends with the total of row r
#pragma unroll 1
        for (int m = 0; m < kFoldChunks; ++m) {
          float dots[kCS];
#pragma unroll
          for (int k = 0; k < kCS; ++k) {
            const int rr = lane / RF::kLpr + RF::kRpi * (kCS * m + k);  // row within the warp's rows
            const float4 sv = *reinterpret_cast<const float4*>(tile + (size_t)rr * N + cf);
            float4 acc = make_float4(fdec * sv.x, fdec * sv.y, fdec * sv.z, fdec * sv.w);
            const float4* cr = reinterpret_cast<const float4*>(coef + (size_t)rr * kStepMaxW);
#pragma unroll
            for (int jj = 0; jj < kStepMaxW / 4; ++jj) {
              const float4 cc = cr[jj];
              const float cs[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float4 b = Bq[4 * jj + e];
                acc.x = fmaf(cs[e], b.x, acc.x);
                acc.y = fmaf(cs[e], b.y, acc.y);
                acc.z = fmaf(cs[e], b.z, acc.z);
                acc.w = fmaf(cs[e], b.w, acc.w);
              }
            }
            const size_t gidx = ((size_t)hg * P + row0 + rr) * N + cf;
            *reinterpret_cast<float4*>(a.S_ckpt + gidx) = acc;
            float4 rdv = acc;  // the row as the decode reads it
            if constexpr (FS == 2) {
              const uint2 pk = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
              *reinterpret_cast<uint2*>(a.S_read + gidx) = pk;
              rdv = make_float4(bf16_lo(pk.x), bf16_hi(pk.x), bf16_lo(pk.y), bf16_hi(pk.y));
            }
            dots[k] = fmaf(rdv.x, c4[0], fmaf(rdv.y, c4[1], fmaf(rdv.z, c4[2], rdv.w * c4[3])));
          }
          const float d = reduce_chunk<RF::kLpr, kCS>(dots, lane);
          if ((lane & (kFoldChunks - 1)) == m) mine = d;
        }
        } else {
        // S' = fold_decay S + c B^T on the tensor cores: mma.sync m16n8k8
        // with TF32 operands split in two (x = hi + lo, three products
        // hi.hi + hi.lo + lo.hi per step: about FP32 accuracy); rows
        // 16 mt + (lane / 4) [+ 8], columns 8 nt + 2 (lane % 4) [+ 1] of each
        // 16 x 8 tile. Then the new rows (as the read copy holds them)
        // dotted with C.
        uint32_t ah[2][2][4], alo[2][2][4];  // c fragments [row tile][entry step][4]
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float v = coef[(size_t)(16 * mt + gq + 8 * (e & 1)) * kStepMaxW + 8 * ks + tq + 4 * (e >> 1)];
              tf32_split(v, ah[mt][ks][e], alo[mt][ks][e]);
            }
        const float* Bg = a.bfold + ((size_t)seq * a.G + g) * kStepMaxW * N;
        const TV* Cg = Cin + ((size_t)seq * a.G + g) * N;
        float racc[2][2] = {};  // [row tile][row, row + 8]: partial dots with C
#pragma unroll 4
        for (int nt = 0; nt < N / 8; ++nt) {
          const int c0 = 8 * nt;
          uint32_t bh[2][2], blo[2][2];  // B fragments [entry step][2] (zero past nf)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int j = 8 * ks + tq + 4 * e;
              const float v = j < nf ? __ldg(Bg + (size_t)j * N + c0 + gq) : 0.f;
              tf32_split(v, bh[ks][e], blo[ks][e]);
            }
          float2 cc;
          if constexpr (sizeof(TV) == 2) {
            const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(Cg + c0 + 2 * tq));
            cc = make_float2(bf16_lo(w), bf16_hi(w));
          } else {
            cc = __ldg(reinterpret_cast<const float2*>(Cg + c0 + 2 * tq));
          }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const int ra = 16 * mt + gq;
            const float2 s0 = *reinterpret_cast<const float2*>(tile + (size_t)ra * N + c0 + 2 * tq);
            const float2 s1 = *reinterpret_cast<const float2*>(tile + (size_t)(ra + 8) * N + c0 + 2 * tq);
            float d[4] = {fdec * s0.x, fdec * s0.y, fdec * s1.x, fdec * s1.y};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              mma_tf32(d, ah[mt][ks], bh[ks][0], bh[ks][1]);
              mma_tf32(d, ah[mt][ks], blo[ks][0], blo[ks][1]);
              mma_tf32(d, alo[mt][ks], bh[ks][0], bh[ks][1]);
            }
            const size_t g0 = ((size_t)hg * P + row0 + ra) * N + c0 + 2 * tq, g1 = g0 + (size_t)8 * N;
            *reinterpret_cast<float2*>(a.S_ckpt + g0) = make_float2(d[0], d[1]);
            *reinterpret_cast<float2*>(a.S_ckpt + g1) = make_float2(d[2], d[3]);
            float2 r0v = make_float2(d[0], d[1]), r1v = make_float2(d[2], d[3]);
            if constexpr (FS == 2) {
              const uint32_t p0 = pack_bf16x2(d[0], d[1]), p1 = pack_bf16x2(d[2], d[3]);
              *reinterpret_cast<uint32_t*>(a.S_read + g0) = p0;
              *reinterpret_cast<uint32_t*>(a.S_read + g1) = p1;
              r0v = make_float2(bf16_lo(p0), bf16_hi(p0));
              r1v = make_float2(bf16_lo(p1), bf16_hi(p1));
            }
            racc[mt][0] = fmaf(r0v.x, cc.x, fmaf(r0v.y, cc.y, racc[mt][0]));
            racc[mt][1] = fmaf(r1v.x, cc.x, fmaf(r1v.y, cc.y, racc[mt][1]));
          }
        }
        // totals over the four lanes of a row group; lane (gq, tq) keeps row r
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            racc[mt][h2] += __shfl_xor_sync(kFull, racc[mt][h2], 1);
            racc[mt][h2] += __shfl_xor_sync(kFull, racc[mt][h2], 2);
          }
        mine = (tq & 2) ? ((tq & 1) ? racc[1][1] : racc[1][0])
                        : ((tq & 1) ? racc[0][1] : racc[0][0]);
        }
        yrow[r] = fmaf(scale, mine, extra);
        rxh[(size_t)tslot * P + r] = xtr;  // append the token's x
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty[s0]);
          if (FS > 1) mbar_arrive(&empty[s1]);
        }
      }
    }
  }
  __syncthreads();
  // The block's units are done: one arrival per unit on its sequence's
  // counter; the last of a sequence's H * nrb arrivals moves its pointers.
  // No fence: the pointers the last arrival moves are read in this launch
  // only from the block-start tables of blocks that hold units of that
  // sequence (before their own arrivals); the rows and the appended entries
  // only by later launches.
  if (!abort_flag && nloc > tid) {
    for (int i = tid; i < nloc; i += blockDim.x) {
      const int code = table[i];
      if (!(code & 1)) continue;
      const int seq = (b0 + i * G0) / per_seq;
      if (atomicAdd(a.sync + seq, 1) + 1 == per_seq) {
        const int l = (code >> 8) & 0xff, hd = (code >> 16) & 0xff;
        if (code & 2) {
          a.head[seq] = (hd + l) % W;
          a.len[seq] = 1;
        } else {
          a.len[seq] = l + 1;
        }
        a.sync[seq] = 0;
      }
    }
  }
  // No bulk copy may land after the block exits.
  if (tid == 0 && abort_flag) {
    for (int s = 0; s < NS; ++s) {
      mbar_wait(&full[s], 0);
      mbar_wait(&full[s], 1);
    }
  }
}

}  // namespace rs
