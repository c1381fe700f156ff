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
// Units are (sequence, head, row block of RB rows), dealt to the blocks in
// turn (unit u goes to block u mod grid), so the folds of any set of
// sequences spread over all SMs. In each block a producer warp fills a ring
// of NS shared-memory stages with one bulk copy per stage and consumer
// groups of GU warps take the block's units round robin. Two kinds of unit:
//   decode  (ring not full): one stage of read-copy rows;
//           y[r] = decay * (S[r, :] . C) + extra[r]
//   fold    (ring full, n = len entries): FS = 4 / sizeof(TS) stages of FP32
//           checkpoint rows, each with the rows' fold coefficients
//           c_j[r] = w_j x_j[r] (from the preparation grid) beside it;
//           S'[r, :] = fold_decay * S[r, :] + sum_j c_j[r] B_j,
//           S' written to the checkpoint and read copy, then
//           y[r] = decay * (S'_read[r, :] . C) + extra[r]
// where S'_read is the row as the read copy holds it (the BF16 rounding when
// there is one), so outputs equal those of a consolidate then a decode.
// The kind of every unit is fixed at block start from the ring pointers,
// which nothing changes until the last unit of a sequence is done: each
// block arrives on a sequence's counter once per unit of it when all its
// units are done, and the last arrival moves the pointers (fold:
// head += len, len = 1; else len += 1).
//
// Stages are used in unit order (a fold unit takes FS consecutive ones); at
// block start one warp numbers them, so each unit's entry holds its first
// stage and that fill's mbarrier parity. The producer streams
// read-copy rows before the preparation grid ends, but waits for it before
// the first fold unit (whose coefficients that grid writes).
#pragma once

#include "common.cuh"
#include "launch.h"
#include "stream.cuh"

namespace rs {

struct StepArgs {
  int batch, H, G, P, W, RB, nrb, NS, GU, nloc_max;
  const void* S;        // decode rows: the read copy, or the checkpoint without one
  float* S_ckpt;        // FP32 checkpoint [b, H, P, N]
  bf16* S_read;         // BF16 read copy or null
  float* out;           // y [b, H, P]
  const float* work;    // rows of wrow floats per (sequence, head), StepLayout
  int wrow;
  const float* pack;    // fold coefficients [b, H, P, kStepMaxW]
  const float* bfold;   // folded B rows [b, G, kStepMaxW, N]
  const void* C;        // [b, G, N]
  int32_t* head;
  int32_t* len;
  int32_t* status;
  int32_t* sync;
};

// Shared memory: NS stages, NS coefficient side buffers, full and empty
// barriers, and the kind of each of the block's units.
struct StepSmem {
  size_t stage, side, sides, bars, table, total;
  __host__ __device__ StepSmem(int RB, int N, int ts, int NS, int nloc_max) {
    stage = stream_stage_bytes(RB, N, ts);
    side = (size_t)(RB / (4 / ts)) * kStepMaxW * 4;  // coefficients of a stage's FP32 rows
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

template <int N, typename TS, typename TV>
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
  const StepSmem L(RB, N, sizeof(TS), NS, a.nloc_max);
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
  const uint32_t side_bytes = (uint32_t)L.side;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], GU);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  // Each local unit's entry: bit 0 pointers valid, bit 1 fold, its first
  // stage in bits 2..6 and that fill's mbarrier parity in bit 7, len in bits
  // 8..15, head in bits 16..23. The kinds first, then one warp numbers the
  // stages in unit order (a fold unit takes FS of them).
  for (int i = tid; i < nloc; i += blockDim.x) {
    const int seq = (b0 + i * G0) / per_seq;
    const int l = a.len[seq], hd = a.head[seq];
    const bool ok = pointers_ok(hd, l, W);
    const bool fold = ok && l + 1 > W;
    table[i] = (ok ? 1 : 0) | (fold ? 2 : 0) | (ok ? (l << 8) | (hd << 16) : 0);
  }
  __syncthreads();
  if (warp == 0) {
    int base = 0;  // stages of the units before this chunk of 32
    for (int i0 = 0; i0 < nloc; i0 += 32) {
      const int i = i0 + lane;
      const int e = i < nloc ? table[i] : 0;
      const int n = i < nloc ? ((e & 2) ? FS : 1) : 0;
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
      }
      const int c = base + incl - n;  // stages before unit i
      if (i < nloc) table[i] = e | ((c % NS) << 2) | (((c / NS) & 1) << 7);
      base += __shfl_sync(kFull, incl, 31);
    }
  }
  __syncthreads();

  if (warp == CW) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_evict_first_policy();
    const TS* Sg = reinterpret_cast<const TS*>(a.S);
    int s = 0;           // stage of the next fill
    uint32_t ph = 0;     // parity of that fill (the previous fill of the stage: ph ^ 1)
    bool reuse = false;  // the stages are being refilled
    bool stop = false, prep_done = false;
    for (int i = 0; i < nloc && !stop; ++i) {
      const int u = b0 + i * G0;
      const int hg = nrb == 1 ? u : u / nrb, rb = u - hg * nrb;
      const bool fold = (table[i] & 2) != 0;
      if (fold && !prep_done) {  // the coefficients come from the preparation grid
        griddep_wait();
        prep_done = true;
      }
      const int nst = fold ? FS : 1;
      for (int f = 0; f < nst; ++f) {
        if (reuse && !mbar_wait_warp(&empty[s], ph ^ 1)) {
          if (lane == 0) abort_flag = 1;
          stop = true;
          break;
        }
        if (lane == 0) {
          const size_t row = (size_t)hg * P + (size_t)rb * RB;
          if (fold) {
            const size_t r0 = row + (size_t)f * (RB / FS);
            mbar_arrive_expect_tx(&full[s], tile_bytes + side_bytes);
            bulk_g2s(smem + (size_t)s * L.stage, a.S_ckpt + r0 * N, tile_bytes, &full[s], pol);
            bulk_g2s(smem + L.sides + (size_t)s * L.side, a.pack + r0 * kStepMaxW, side_bytes,
                     &full[s]);
          } else {
            mbar_arrive_expect_tx(&full[s], tile_bytes);
            bulk_g2s(smem + (size_t)s * L.stage, Sg + row * N, tile_bytes, &full[s], pol);
          }
        }
        if (++s == NS) {
          s = 0;
          ph ^= 1;
          reuse = true;
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
    // Work rows and folded B rows come from the preparation grid (this grid
    // may start before it ends).
    griddep_wait();
    for (int i = gi; i < nloc; i += NG) {
      const int u = b0 + i * G0;
      const int hg = nrb == 1 ? u : u / nrb, rb = u - hg * nrb;
      const int seq = hg / H, h = hg - seq * H;
      const int g = h / (H / a.G);
      const int code = table[i];
      const bool ok = (code & 1) != 0, fold = (code & 2) != 0;
      const int s0 = (code >> 2) & 31;            // the unit's first stage
      const uint32_t ph0 = (code >> 7) & 1;       // and the parity of its fill
      const int row0 = rb * RB + part * RBp;  // first row of this warp within the head
      const float* w0 = a.work + (size_t)hg * a.wrow;
      float* yrow = a.out + (size_t)hg * P + row0;
      const float scale = w0[P];
      const bool aborted = __shfl_sync(kFull, abort_flag, 0) != 0;
      if (!fold) {
        // -------------------------------------------------- decode unit
        float vec[kE];
        load_vec<TV, kE>(Cin + ((size_t)seq * a.G + g) * N + cd, vec);
        const float extra = w0[row0 + RD::row_of(lane)];
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
        if (ok) yrow[RD::row_of(lane)] = fmaf(scale, d, extra);
      } else {
        // ---------------------------------------------------- fold unit
        const int nf = (code >> 8) & 0xff;
        const float fdec = w0[P + 1];
        // B_j of the head's group, this lane's columns (zero past the n entries)
        const float* Bs = a.bfold + ((size_t)seq * a.G + g) * kStepMaxW * N + cf;
        float4 Bq[kStepMaxW];
#pragma unroll
        for (int j = 0; j < kStepMaxW; ++j)
          Bq[j] = j < nf ? *reinterpret_cast<const float4*>(Bs + (size_t)j * N)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        float c4[4];
        load_vec<TV, 4>(Cin + ((size_t)seq * a.G + g) * N + cf, c4);
        const int r = fold_row<RF::kLpr, RF::kRpi, kCS>(lane);
        const float extra = w0[row0 + r];
        // this warp's stage: the unit's first, or for the second half of a
        // two-stage unit the next one (wrapping flips the parity)
        const bool second = FS > 1 && part == 1;
        const bool wrap = second && s0 + 1 == NS;
        const int s = second ? (wrap ? 0 : s0 + 1) : s0;
        const bool landed = !aborted && mbar_wait_warp(&full[s], wrap ? ph0 ^ 1 : ph0);
        if (!aborted && !landed && lane == 0) {
          abort_flag = 1;
          atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
        }
        if (group_any(!landed)) break;
        // this warp's 32 FP32 rows and their coefficients
        const int off = FS > 1 ? 0 : part * RBp;
        const float* tile = reinterpret_cast<const float*>(smem + (size_t)s * L.stage) + (size_t)off * N;
        const float* coef = reinterpret_cast<const float*>(smem + L.sides + (size_t)s * L.side) +
                            (size_t)off * kStepMaxW;
        // rows in chunks of kCS per lane; lane l ends with the total of row r
        float mine = 0.f;
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
        yrow[r] = fmaf(scale, mine, extra);
        __syncwarp();
        if (lane == 0)
          for (int f = 0; f < FS; ++f) mbar_arrive(&empty[s0 + f < NS ? s0 + f : s0 + f - NS]);
      }
    }
  }
  __syncthreads();
  // The block's units are done: one arrival per unit on its sequence's
  // counter (one fence per thread); the last of a sequence's H * nrb
  // arrivals moves its pointers.
  if (!abort_flag && nloc > tid) {
    __threadfence();
    for (int i = tid; i < nloc; i += blockDim.x) {
      const int code = table[i];
      if (!(code & 1)) continue;
      const int seq = (b0 + i * G0) / per_seq;
      if (atomicAdd(a.sync + seq, 1) + 1 == per_seq) {
        __threadfence();
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
