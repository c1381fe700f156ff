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
// S_c once for all drafts. Decode and verify are one persistent kernel whose
// prep warps run the sweeps while its producer and consumer warps stream S_c
// and write o = S_c u + buffer terms for every query. The fold applies the n updates
// row by row in FP32 registers: s <- alpha (.) s; s <- s + beta (v_r - s.k) k.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>

#include "common.cuh"
#include "launch.h"

namespace rs {
namespace {

// ------------------------------------------------------ Gram form of the sweeps

constexpr int kGramN = 16;     // entries of one Gram tile
constexpr int kGramQ = 8;      // queries of one Gram tile (the n = 8 columns)
constexpr int kGramT = 24;     // floats per scratch row: G[j][0..15], P[j][0..7]

// Gram form of the backward sweeps of one head (GDN). With G[j][i] = k_j . k_i
// and P[j][t] = scale k_j . q_t, the sweep of query t (entries top = len + t
// down to 0) keeps a[j] = k_j . u for every j below the current entry: it
// starts at P[j][t], and entry i (c_i = beta_i a[i]) turns it into
//   a[j] <- alpha_i (a[j] - c_i G[j][i]),
// since u <- alpha_i (u - c_i k_i). So the coefficients c come from scalar
// updates instead of n dot products over d_k, each behind a warp reduction.
// G and P are one tensor-core tile: mma.sync m16n8k16 on the BF16 k rows
// (exact products, FP32 sums), the k rows doubling as the B operand of G
// (rows past n repeat row n - 1 and queries past K are zero, so every entry
// of the tile is finite and the unused ones are never selected). Lane j
// holds a[j] of every query; entry i broadcasts a[i] with one shuffle per
// query, so the queries' chains interleave. c[t][i] goes to c_out.
template <int DK, int KMAX>
__device__ __forceinline__ void gram_coefficients(const unsigned char* kbase, const unsigned char* qbase,
                                                  uint32_t ks, const float* ar, const float* br, int len,
                                                  int K, float scale, float* __restrict__ T,
                                                  float* __restrict__ c_out, int lane) {
  const int g = lane >> 2, t4 = lane & 3;
  float dg0[4] = {0.f, 0.f, 0.f, 0.f}, dg1[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
  // ldmatrix row addresses: matrix m = lane / 8 covers row (m & 1) * 8 + lane % 8
  // and the column half m >> 1 of each 16-column step
  const int m = lane >> 3, n = len + K;
  const int row = min((m & 1) * 8 + (lane & 7), n - 1);
  const uint32_t a_addr = smem_u32(kbase) + row * ks + (m >> 1) * 16;
  // query B fragments straight from the q rows: column g = query g
  const uint32_t* qw = reinterpret_cast<const uint32_t*>(qbase + (g < K ? g : 0) * ks) + t4;
  uint32_t a[DK / 16][4], b[DK / 16][2];
#pragma unroll
  for (int kk = 0; kk < DK / 16; ++kk) {
    ldsm_x4(a[kk], a_addr + kk * 32);
    b[kk][0] = g < K ? qw[kk * 8] : 0u;
    b[kk][1] = g < K ? qw[kk * 8 + 4] : 0u;
  }
#pragma unroll
  for (int kk = 0; kk < DK / 16; ++kk) {
    mma_bf16_16816(dg0, a[kk], a[kk][0], a[kk][2]);  // columns: k rows 0-7
    mma_bf16_16816(dg1, a[kk], a[kk][1], a[kk][3]);  // k rows 8-15
    mma_bf16_16816(dp, a[kk], b[kk][0], b[kk][1]);   // queries 0-7
  }
  *reinterpret_cast<float2*>(T + g * kGramT + 2 * t4) = make_float2(dg0[0], dg0[1]);
  *reinterpret_cast<float2*>(T + (g + 8) * kGramT + 2 * t4) = make_float2(dg0[2], dg0[3]);
  *reinterpret_cast<float2*>(T + g * kGramT + 8 + 2 * t4) = make_float2(dg1[0], dg1[1]);
  *reinterpret_cast<float2*>(T + (g + 8) * kGramT + 8 + 2 * t4) = make_float2(dg1[2], dg1[3]);
  *reinterpret_cast<float2*>(T + g * kGramT + 16 + 2 * t4) = make_float2(dp[0], dp[1]);
  *reinterpret_cast<float2*>(T + (g + 8) * kGramT + 16 + 2 * t4) = make_float2(dp[2], dp[3]);
  __syncwarp();
  const int j = lane & (kGramN - 1);
  float acc[KMAX];
#pragma unroll
  for (int t = 0; t < KMAX; ++t) acc[t] = t < K ? scale * T[j * kGramT + 16 + t] : 0.f;
  for (int i = n - 1; i >= 0; --i) {
    const float gji = T[j * kGramT + i], bi = br[i], ai = ar[i];
#pragma unroll
    for (int t = 0; t < KMAX; ++t) {
      const float s = __shfl_sync(kFull, acc[t], i);
      const bool vis = t < K && i <= len + t;  // entry i is below query t's top
      const float c = vis ? bi * s : 0.f;
      if (vis && lane == 0) c_out[t * kGramN + i] = c;
      acc[t] = vis && j < i ? ai * fmaf(-c, gji, acc[t]) : acc[t];
    }
  }
  __syncwarp();
}

// ------------------------------------------------------ fused decode / verify

constexpr int kFGroups = 4;    // consumer groups
constexpr int kFWarps = 16;    // warps per block: consumers, the producer, prep warps
constexpr int kFQ = 4;         // queries swept together (verify); decode sweeps one
constexpr int kFMaxSlots = 16; // per-head vector slots between prep and consumers

struct DFused {
  int batch, H, DV, W, K, commit;  // K queries per head; commit: decode (len += 1)
  int RB, nrb, NS, GU;             // rows per unit, units per head, stages, warps per group
  int NP, depth, NSL;              // prep warps, heads in flight per prep warp, vector slots
  const void* S;                   // state rows [b, H, DV, DK] (read copy or checkpoint)
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  float scale;
  float* o;                        // [b, K, H, DV]
  void* ring_q;
  void* ring_k;
  void* ring_v;
  float* ring_alpha;
  float* ring_beta;
  int32_t* head;
  int32_t* len;
  int32_t* status;
  int32_t* sync;
  // fused fold + decode step only (else null): a sequence whose ring is full
  // is not refused but left to the fold grid that follows, which decodes its
  // token from the folded rows; flags[seq] = 1 marks it, 0 any other
  int32_t* flags;
};

// One head stage of a prep warp (byte offsets): a header (len, head, ok),
// then the entries 0..n-1 in order (k rows, v rows, gates, beta) and the K
// queries.
struct DStage {
  size_t kr, vr, ar, br, qr, bytes;
  __host__ __device__ DStage(int DK, int DV, int W, int K, bool kda, int ti) {
    kr = 16;                                                     // [W][DK] k_j (in_dtype)
    vr = kr + align_up((size_t)W * DK * ti, 16);                 // [W][DV] v_j (in_dtype)
    ar = vr + align_up((size_t)W * DV * ti, 16);                 // KDA [W][DK], GDN [W]
    br = ar + align_up((size_t)W * (kda ? DK : 1) * 4, 16);      // [W] beta_j
    qr = br + align_up((size_t)W * 4, 16);                       // [K][DK] q_i (in_dtype)
    bytes = align_up(qr + (size_t)K * DK * ti, 128);
  }
};

// Shared memory of the fused block: NS state stages and their barriers, NSL
// vector slots (u[K][DK], e[K][DV], ok) and their barriers, then NP prep
// warps with `depth` head stages each.
struct DFusedSmem {
  size_t stage, bars, slot, slots, vbars, prep, prep_warp, total;
  __host__ __device__ DFusedSmem(int RB, int DK, int DV, int W, int K, int NS, int NSL, int NP,
                                 int depth, bool kda, int ts, int ti) {
    stage = align_up((size_t)RB * DK * ts, 128);
    bars = (size_t)NS * stage;
    slots = align_up(bars + 16 * (size_t)NS, 128);
    slot = align_up((size_t)K * (DK + DV) * 4 + 16, 128);
    vbars = slots + (size_t)NSL * slot;
    prep = align_up(vbars + 16 * (size_t)NSL, 128);
    prep_warp = (size_t)depth * DStage(DK, DV, W, K, kda, ti).bytes;
    total = prep + (size_t)NP * prep_warp;
  }
};

// Replay decode (K = 1, commits the token) or speculative verify (K drafts,
// commits nothing) of the delta-rule layers in one persistent kernel; one
// block per SM owns a contiguous range of heads (flat index seq * H + h),
// split in units of RB state rows.
//
// Prep warps (NP) take the block's heads round robin. For a head they stage
// its entries with async copies (`depth` heads ahead): entry j < len is ring
// slot (head + j) mod W, entry len + i is the call's input i. For query i
// (entry len + i; drafts 0..i visible) the backward sweep over entries
// len+i..0 is
//   u <- scale q_i; for j: s = k_j . u; c = beta_j s; e_i += c v_j;
//   u <- alpha_j (.) (u - c k_j)
// (queries swept together share each entry's loads). u and e go to the
// head's vector slot. The warp appends the call's entries to slots
// (head + len + i) mod W and, for a decode, arrives once per sequence on its
// arrival counter (the last arrival bumps len). A sequence without room for K
// entries (or with pointers out of range) gets a status bit and no output.
//
// The producer warp streams the state rows unit by unit with bulk copies into
// NS stages while consumer groups of GU warps take units round robin and
// write o_i[r] = S[r, :] . u_i + e_i[r] from the slot. The state is read once
// for all queries. Every wait is bounded; a timeout sets
// REPLAYSSM_SEQ_TIMEOUT and ends the block.
template <int DK, typename TS, typename TI, bool KDA, int KMAX>
__global__ void __launch_bounds__(32 * kFWarps, 1) delta_fused_kernel(const DFused a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using RD = RowDot<DK, TS>;
  constexpr int kE = RD::kEpc;
  constexpr int KQ = KMAX == 1 ? 1 : kFQ;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int GU = a.GU, CW = kFGroups * GU, NG = kFGroups, NS = a.NS, NSL = a.NSL;
  const int H = a.H, DV = a.DV, RB = a.RB, nrb = a.nrb, K = a.K, W = a.W;
  const DFusedSmem L(RB, DK, DV, W, K, NS, NSL, a.NP, a.depth, KDA, sizeof(TS), sizeof(TI));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + NS;
  uint64_t* vfull = reinterpret_cast<uint64_t*>(smem + L.vbars);
  uint64_t* vempty = vfull + NSL;
  __shared__ int abort_smem;
  volatile int& abort_flag = abort_smem;
  const long long heads = (long long)a.batch * H;
  const int hb0 = (int)(heads * blockIdx.x / gridDim.x);
  const int hb1 = (int)(heads * (blockIdx.x + 1) / gridDim.x);
  const int nh = hb1 - hb0, nu = nh * nrb;
  const uint32_t tile_bytes = (uint32_t)((size_t)RB * DK * sizeof(TS));
  // slot layout (floats): u [K][DK], e [K][DV], then the ok flag
  auto slot_ptr = [&](int li) {
    return reinterpret_cast<float*>(smem + L.slots + (size_t)(li % NSL) * L.slot);
  };
  const int ok_off = K * (DK + DV);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], GU);
    }
    for (int s = 0; s < NSL; ++s) {
      mbar_init(&vfull[s], 32);
      mbar_init(&vempty[s], nrb * GU);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  // (A fused step's fold grid is this grid's programmatic dependent. No early
  // trigger: it launches as this grid completes, its launch overlapping the
  // completion, and waits with griddepcontrol.wait before it reads the flags
  // and pointers. Triggered at the start, its blocks queued behind this
  // grid's and the staggered steps, which fold in every call, got slower.)
  // The sequences of this block's heads that are refused (pointers out of
  // range, or no room for K entries: with a.flags, the full rings left to
  // the fold grid): their state rows are not read. Read here, before any
  // prep warp of this block runs, so before the last arrival of any of
  // those sequences can move its pointers (it needs this block's heads).
  // Ranges of more than kSkipSeqs sequences stream every head.
  constexpr int kSkipSeqs = 1024;
  __shared__ uint32_t skipmask[kSkipSeqs / 32];
  const int seq_lo = hb0 / H, nseq = nh > 0 ? (hb1 - 1) / H - seq_lo + 1 : 0;
  const bool use_skip = nseq <= kSkipSeqs;
  for (int i = tid; i < kSkipSeqs / 32; i += blockDim.x) skipmask[i] = 0u;
  __syncthreads();
  if (use_skip) {
    for (int i = tid; i < nseq; i += blockDim.x) {
      const int l = a.len[seq_lo + i], hd = a.head[seq_lo + i];
      if (!pointers_ok(hd, l, W) || l + K > W) atomicOr(&skipmask[i / 32], 1u << (i % 32));
    }
  }
  __syncthreads();

  if (warp == CW) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_evict_first_policy();
    const TS* Sg = reinterpret_cast<const TS*>(a.S);
    int ps = 0;
    uint32_t pk = 0;
    bool pwrap = false;
    int li = 0, rb = 0;
    bool skip = false;  // the current head's sequence is refused or left to the fold
    for (int ul = 0; ul < nu; ++ul) {
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
      if (rb == 0) {
        // a refused head's stages complete without data: its rows are not
        // needed and not read from memory
        const int i = (hb0 + li) / H - seq_lo;
        skip = use_skip && ((skipmask[i / 32] >> (i % 32)) & 1u) != 0;
      }
      if (lane == 0) {
        if (skip) {
          mbar_arrive(&full[s]);
        } else {
          mbar_arrive_expect_tx(&full[s], tile_bytes);
          bulk_g2s(smem + (size_t)s * L.stage,
                   Sg + ((size_t)(hb0 + li) * DV + (size_t)rb * RB) * DK, tile_bytes, &full[s], pol);
        }
      }
      if (++rb == nrb) {
        rb = 0;
        ++li;
      }
    }
  } else if (warp < CW) {
    // ------------------------------------------------------------ consumers
    const int gi = warp / GU, part = warp - gi * GU;
    const int RBp = RB / GU;
    const int ngr = RBp / 32;
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
    const int c0 = RD::chunk_of(lane) * kE;
    int s = gi;
    uint32_t ph = 0;
    for (int ul = gi; ul < nu; ul += NG) {
      const int li = ul / nrb, rb = ul - li * nrb;
      const int hg = hb0 + li, seq = hg / H, h = hg - seq * H;
      const int row0 = rb * RB + part * RBp;
      const bool aborted0 = __shfl_sync(kFull, abort_flag, 0) != 0;
      const bool vready = !aborted0 && mbar_wait_warp(&vfull[li % NSL], (li / NSL) & 1);
      if (!aborted0 && !vready && lane == 0) {
        abort_flag = 1;
        atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
      }
      if (group_any(!vready)) break;
      const float* sl = slot_ptr(li);
      const bool write = reinterpret_cast<const int*>(sl)[ok_off] != 0;
      float vec[KMAX][kE];
      float extra[4];
#pragma unroll
      for (int kq = 0; kq < KMAX; ++kq) {
        if (kq >= K) break;
#pragma unroll
        for (int e = 0; e < kE; e += 4) {
          const float4 v4 = *reinterpret_cast<const float4*>(sl + kq * DK + c0 + e);
          vec[kq][e] = v4.x;
          vec[kq][e + 1] = v4.y;
          vec[kq][e + 2] = v4.z;
          vec[kq][e + 3] = v4.w;
        }
      }
      if constexpr (KMAX == 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < ngr) extra[q] = sl[K * DK + row0 + 32 * q + RD::row_of(lane)];
      }
      const bool aborted = __shfl_sync(kFull, abort_flag, 0) != 0;
      const bool landed = !aborted && mbar_wait_warp(&full[s], ph);
      if (!aborted && !landed && lane == 0) {
        abort_flag = 1;
        atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
      }
      if (group_any(!landed)) break;
      const TS* tile = reinterpret_cast<const TS*>(smem + (size_t)s * L.stage) + (size_t)part * RBp * DK;
      float* yrow = a.o + ((size_t)seq * K * H + h) * DV + row0;
      if constexpr (KMAX > 1) {
        constexpr int KC = KMAX < 64 / RD::kLpr ? KMAX : 64 / RD::kLpr;
#pragma unroll 1
        for (int q = 0; q < ngr; ++q) {
          if (!write) break;  // (a refused head's stage holds no rows)
          const int r = 32 * q + RD::row_of(lane);
#pragma unroll 1
          for (int k0 = 0; k0 < KMAX; k0 += KC) {
            if (k0 >= K) break;
            float ex[KC];
#pragma unroll
            for (int c = 0; c < KC; ++c) ex[c] = k0 + c < K ? sl[K * DK + (k0 + c) * DV + row0 + r] : 0.f;
            float acc[KC][RD::kLpr];
            const TS* base = tile + (size_t)(32 * q + lane / RD::kLpr) * DK + c0;
#pragma unroll
            for (int kk = 0; kk < RD::kLpr; ++kk) {
              const uint4 raw = *reinterpret_cast<const uint4*>(base + (size_t)kk * RD::kRpi * DK);
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
              if (write) yrow[(size_t)(k0 + c) * H * DV + r] = d + ex[c];
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty[s]);
          mbar_arrive(&vempty[li % NSL]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q >= ngr || !write) break;  // (a refused head's stage holds no rows)
          const float d = RD::rows32(tile, 32 * q, vec[0], lane);
          yrow[32 * q + RD::row_of(lane)] = d + extra[q];
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty[s]);
          mbar_arrive(&vempty[li % NSL]);
        }
      }
      s += NG;
      if (s >= NS) {
        s -= NS;
        ph ^= 1;
      }
    }
  } else if (warp - CW - 1 < a.NP) {
    // ------------------------------------------------------------ prep
    constexpr int EPL = DK / 32;
    constexpr int ti = (int)sizeof(TI);
    constexpr int kKC = DK * ti / 16;  // 16-byte chunks of a k row (<= 32)
    constexpr int kKR = 32 / kKC;
    constexpr int kAC = DK * 4 / 16;   // chunks of a KDA gate row
    constexpr int kAR = 32 / kAC;
    const int NP = a.NP, depth = a.depth;
    const int pw = warp - CW - 1;
    const int Wd = ring_wd(W);
    const DStage SL(DK, DV, W, K, KDA, ti);
    unsigned char* wbase = smem + L.prep + (size_t)pw * L.prep_warp;
    const size_t krow = (size_t)DK * ti, arow = (size_t)DK * 4, vrow = (size_t)DV * ti;
    const int vcpr = (int)(vrow / 16);  // 16-byte chunks of a v row
    const bool vmap = vcpr <= 32 && 32 % vcpr == 0;
    const int vro = vmap ? lane / vcpr : 0, vch = vmap ? lane - vro * vcpr : 0;
    const int vstep = vmap ? 32 / vcpr : 0;
    const int EVL = DV / 32;            // e rows per lane: r = lane + 32 m
    const int nmine = nh > pw ? (nh - pw + NP - 1) / NP : 0;  // heads of this warp

    // ---- issue side: stage the entries of this warp's head i_t
    int i_t = 0, i_loaded = -1, i_len = 0, i_hd = 0;
    bool i_ok = false;
    int i_v = hb0 + pw, i_seq = i_v / H, i_h = i_v - (i_v / H) * H;
    auto issue = [&]() {
      if (i_seq != i_loaded) {
        int l = 0, hh = 0;
        if (lane == 0) {
          l = a.len[i_seq];
          hh = a.head[i_seq];
        }
        i_len = __shfl_sync(kFull, l, 0);
        i_hd = __shfl_sync(kFull, hh, 0);
        i_ok = pointers_ok(i_hd, i_len, W) && i_len + K <= W;
        i_loaded = i_seq;
      }
      unsigned char* st = wbase + (size_t)(i_t % depth) * SL.bytes;
      if (lane == 0) {
        int* hdr = reinterpret_cast<int*>(st);
        hdr[0] = i_len;
        hdr[1] = i_hd;
        hdr[2] = i_ok ? 1 : 0;
        hdr[3] = i_seq;
      }
      if (i_ok) {
        const int n = i_len + K, v = i_v;
        const size_t in0 = (size_t)i_seq * K * H + i_h;  // input row of draft 0 ([b, K, H])
        const size_t instep = (size_t)H;                 // rows between drafts
        {
          const unsigned char* rkh = reinterpret_cast<const unsigned char*>(a.ring_k) + (size_t)v * W * krow;
          const unsigned char* ikh = reinterpret_cast<const unsigned char*>(a.k) + in0 * krow;
          const int c = (lane % kKC) * 16;
          for (int j = lane / kKC; j < n; j += kKR) {
            const int slot = i_hd + j < W ? i_hd + j : i_hd + j - W;
            const unsigned char* src = j < i_len ? rkh + slot * krow : ikh + (size_t)(j - i_len) * instep * krow;
            cp_async16(st + SL.kr + j * krow + c, src + c);
          }
          const unsigned char* iqh = reinterpret_cast<const unsigned char*>(a.q) + in0 * krow;
          for (int i = lane / kKC; i < K; i += kKR)
            cp_async16(st + SL.qr + i * krow + c, iqh + (size_t)i * instep * krow + c);
        }
        {
          const unsigned char* rvh = reinterpret_cast<const unsigned char*>(a.ring_v) + (size_t)v * W * vrow;
          const unsigned char* ivh = reinterpret_cast<const unsigned char*>(a.v) + in0 * vrow;
          if (vmap) {
            for (int j = vro; j < n; j += vstep) {
              const int slot = i_hd + j < W ? i_hd + j : i_hd + j - W;
              const unsigned char* src = j < i_len ? rvh + slot * vrow : ivh + (size_t)(j - i_len) * instep * vrow;
              cp_async16(st + SL.vr + j * vrow + vch * 16, src + vch * 16);
            }
          } else {
            for (int idx = lane; idx < n * vcpr; idx += 32) {
              const int j = idx / vcpr, c = idx - j * vcpr;
              const int slot = i_hd + j < W ? i_hd + j : i_hd + j - W;
              const unsigned char* src = j < i_len ? rvh + slot * vrow : ivh + (size_t)(j - i_len) * instep * vrow;
              cp_async16(st + SL.vr + j * vrow + c * 16, src + c * 16);
            }
          }
        }
        if (KDA) {
          const unsigned char* rah = reinterpret_cast<const unsigned char*>(a.ring_alpha) + (size_t)v * W * arow;
          const unsigned char* iah = reinterpret_cast<const unsigned char*>(a.alpha) + in0 * arow;
          const int c = (lane % kAC) * 16;
          for (int j = lane / kAC; j < n; j += kAR) {
            const int slot = i_hd + j < W ? i_hd + j : i_hd + j - W;
            const unsigned char* src = j < i_len ? rah + slot * arow : iah + (size_t)(j - i_len) * instep * arow;
            cp_async16(st + SL.ar + j * arow + c, src + c);
          }
        }
        if (lane < n) {
          const int j = lane;
          const int slot = i_hd + j < W ? i_hd + j : i_hd + j - W;
          const size_t rs_ = (size_t)v * Wd + slot, is_ = in0 + (size_t)(j - i_len) * instep;
          cp_async4(st + SL.br + 4 * j, j < i_len ? a.ring_beta + rs_ : a.beta + is_);
          if (!KDA) cp_async4(st + SL.ar + 4 * j, j < i_len ? a.ring_alpha + rs_ : a.alpha + is_);
        }
        if (lane + 32 < n) {  // windows above 32 entries
          const int j = lane + 32;
          const int slot = i_hd + j < W ? i_hd + j : i_hd + j - W;
          const size_t rs_ = (size_t)v * Wd + slot, is_ = in0 + (size_t)(j - i_len) * instep;
          cp_async4(st + SL.br + 4 * j, j < i_len ? a.ring_beta + rs_ : a.beta + is_);
          if (!KDA) cp_async4(st + SL.ar + 4 * j, j < i_len ? a.ring_alpha + rs_ : a.alpha + is_);
        }
      }
      cp_async_commit();  // one group per head (possibly empty)
      ++i_t;
      i_v += NP;
      i_h += NP;
      while (i_h >= H) {
        i_h -= H;
        ++i_seq;
      }
    };

    // ---- arrivals: a decode's last arrival on a sequence's counter commits
    // len + 1. Lane 0 adds its heads' count and looks at the count it got back
    // at its next arrival, so the atomic's round trip is off the warp's path.
    // No fence: len is read in this launch only at block start and by warps
    // that have not yet arrived for that sequence; the appended ring entries
    // only by later launches.
    int pend_seq = -1, pend_old = 0, pend_units = 0, pend_len = 0;
    auto settle = [&]() {
      if (pend_seq >= 0 && pend_old + pend_units == H) {
        a.len[pend_seq] = pend_len;
        a.sync[pend_seq] = 0;
      }
      pend_seq = -1;
    };
    auto arrive_seq = [&](int sq, int units, int new_len) {
      settle();
      pend_seq = sq;
      pend_units = units;
      pend_len = new_len;
      pend_old = atomicAdd(a.sync + sq, units);
    };

    // ---- compute side
    int cur_seq = -1, len = 0, hd = 0, seq_count = 0;
    bool ok = false;
    int h = (hb0 + pw) % H;
    while (i_t < depth - 1 && i_t < nmine) issue();
    for (int t = 0; t < nmine; ++t) {
      if (i_t < nmine) {
        issue();
        if (depth == 2)
          cp_async_wait_group<1>();  // head t has landed
        else
          cp_async_wait_all();
      } else {
        cp_async_wait_all();
      }
      __syncwarp();
      const int li = pw + t * NP, v = hb0 + li;
      const unsigned char* st = wbase + (size_t)(t % depth) * SL.bytes;
      const int* hdr = reinterpret_cast<const int*>(st);
      const int seq = hdr[3];
      if (seq != cur_seq) {
        if (a.commit && cur_seq >= 0 && ok && lane == 0) arrive_seq(cur_seq, seq_count, len + 1);
        len = hdr[0];
        hd = hdr[1];
        ok = hdr[2] != 0;
        cur_seq = seq;
        seq_count = 0;
        if (h == 0 && lane == 0) {
          const bool deferred = a.flags && !ok && pointers_ok(hd, len, W);  // folds first
          if (a.flags) a.flags[seq] = deferred ? 1 : 0;
          if (!ok && !deferred)
            atomicOr(a.status + seq, pointers_ok(hd, len, W) ? REPLAYSSM_SEQ_RING_FULL
                                                             : REPLAYSSM_SEQ_BAD_POINTER);
        }
      }
      ++seq_count;
      // the slot must have been released by the consumers of head li - NSL
      if (li >= NSL) {
        const bool aborted = __shfl_sync(kFull, abort_flag, 0) != 0;
        const bool freed = !aborted && mbar_wait_warp(&vempty[li % NSL], ((li / NSL) - 1) & 1);
        if (!freed) {
          if (!aborted && lane == 0) {
            abort_flag = 1;
            atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
          }
          break;
        }
      }
      float* sl = slot_ptr(li);
      if (ok) {
        const TI* kr = reinterpret_cast<const TI*>(st + SL.kr);
        const float* ar = reinterpret_cast<const float*>(st + SL.ar);
        const float* br = reinterpret_cast<const float*>(st + SL.br);
        const TI* qr = reinterpret_cast<const TI*>(st + SL.qr);
        const TI* vr = reinterpret_cast<const TI*>(st + SL.vr);
        for (int i0 = 0; i0 < K; i0 += KQ) {
          const int nq = min(KQ, K - i0);
          float u[KQ][EPL], ev[KQ][8];
#pragma unroll
          for (int qi = 0; qi < KQ; ++qi) {
            float qv[EPL];
            load_vec<TI, EPL>(qr + (qi < nq ? i0 + qi : i0) * DK + lane * EPL, qv);
#pragma unroll
            for (int e = 0; e < EPL; ++e) u[qi][e] = qi < nq ? a.scale * qv[e] : 0.f;
#pragma unroll
            for (int m = 0; m < 8; ++m) ev[qi][m] = 0.f;
          }
          const int top = len + i0 + nq - 1;  // newest entry any query of the pass sees
          // entry j's operands, loaded one step ahead
          float kn[EPL], gn[EPL], bn, vn[8];
          auto fetch = [&](int j) {
            load_vec<TI, EPL>(kr + j * DK + lane * EPL, kn);
            if (KDA) {
              load_vec<float, EPL>(ar + j * DK + lane * EPL, gn);
            } else {
              const float g = ar[j];
#pragma unroll
              for (int e = 0; e < EPL; ++e) gn[e] = g;
            }
            bn = br[j];
#pragma unroll
            for (int m = 0; m < 8; ++m) vn[m] = m < EVL ? to_f(vr[j * DV + lane + 32 * m]) : 0.f;
          };
          fetch(top);
          for (int j = top; j >= 0; --j) {
            float kk[EPL], g[EPL], vv[8];
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
              kk[e] = kn[e];
              g[e] = gn[e];
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) vv[m] = vn[m];
            const float bj = bn;
            if (j > 0) fetch(j - 1);
            float sd[KQ];
#pragma unroll
            for (int qi = 0; qi < KQ; ++qi) {
              sd[qi] = 0.f;
#pragma unroll
              for (int e = 0; e < EPL; ++e) sd[qi] = fmaf(kk[e], u[qi][e], sd[qi]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
              for (int qi = 0; qi < KQ; ++qi) sd[qi] += __shfl_xor_sync(kFull, sd[qi], o);
            }
#pragma unroll
            for (int qi = 0; qi < KQ; ++qi) {
              if (qi < nq && j <= len + i0 + qi) {
                const float c = bj * sd[qi];
#pragma unroll
                for (int e = 0; e < EPL; ++e) u[qi][e] = (u[qi][e] - c * kk[e]) * g[e];
#pragma unroll
                for (int m = 0; m < 8; ++m) ev[qi][m] = fmaf(c, vv[m], ev[qi][m]);
              }
            }
          }
#pragma unroll
          for (int qi = 0; qi < KQ; ++qi) {
            if (qi < nq) {
#pragma unroll
              for (int e = 0; e < EPL; ++e) sl[(i0 + qi) * DK + lane * EPL + e] = u[qi][e];
#pragma unroll
              for (int m = 0; m < 8; ++m)
                if (m < EVL) sl[K * DK + (i0 + qi) * DV + lane + 32 * m] = ev[qi][m];
            }
          }
        }
        // append the call's entries: slot (head + len + i) mod W
        for (int i = 0; i < K; ++i) {
          const int j = len + i;
          const int slot = hd + j < W ? hd + j : hd + j - W;
          const size_t rr = (size_t)v * W + slot;
          block_copy_warp(reinterpret_cast<unsigned char*>(a.ring_k) + rr * krow,
                          st + SL.kr + j * krow, (int)krow, lane);
          block_copy_warp(reinterpret_cast<unsigned char*>(a.ring_v) + rr * vrow,
                          st + SL.vr + j * vrow, (int)vrow, lane);
          if (a.ring_q)
            block_copy_warp(reinterpret_cast<unsigned char*>(a.ring_q) + rr * krow,
                            st + SL.qr + i * krow, (int)krow, lane);
          if (KDA)
            block_copy_warp(reinterpret_cast<unsigned char*>(a.ring_alpha) + rr * arow,
                            st + SL.ar + j * arow, (int)arow, lane);
          if (lane == 0) {
            a.ring_beta[(size_t)v * Wd + slot] = br[j];
            if (!KDA) a.ring_alpha[(size_t)v * Wd + slot] = ar[j];
          }
        }
      }
      if (lane == 0) reinterpret_cast<int*>(sl)[ok_off] = ok ? 1 : 0;
      __syncwarp();
      mbar_arrive(&vfull[li % NSL]);  // every lane: its slot writes are released
      h += NP;
      while (h >= H) h -= H;
    }
    cp_async_wait_all();
    if (a.commit && cur_seq >= 0 && ok && lane == 0 && !abort_flag) arrive_seq(cur_seq, seq_count, len + 1);
    if (lane == 0) settle();
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
  // Fused fold + decode step (flags non-null): fold the sequences the decode
  // grid before this one flagged (full rings), then decode their token from
  // the new rows -- o = S' u + ce v with u = A_t (scale q), ce = scale
  // beta (k . q) -- append it (slot head + n) and set len = 1.
  const int32_t* flags;
  const void* q;       // token inputs [b, H, ...]
  const void* k;
  const void* v;
  const float* alpha;  // [b, H] or [b, H, d_k]
  const float* beta;   // [b, H]
  float scale;
  float* o;            // [b, H, d_v]
  void* ring_q;        // optional
  void* ring_kw;       // the same rings, writable
  void* ring_vw;
  float* ring_alphaw;
  float* ring_betaw;
};

// Rows of `cols` elements (in_dtype) of ring entries 0..n-1 of one head --
// entry j is ring slot (head + j) mod W of the head's [W][cols] block -- into
// shared memory as float [n][cols], with 16-byte loads (cols * sizeof(TI)
// a multiple of 16).
template <typename TI>
__device__ __forceinline__ void stage_rows_f32(float* dst, const TI* head_rows, int cols, int n,
                                               int hd, int W) {
  constexpr int epc = 16 / (int)sizeof(TI);  // elements per 16-byte chunk
  const int cpr = cols / epc;
  for (int idx = threadIdx.x; idx < n * cpr; idx += blockDim.x) {
    const int j = idx / cpr, c = idx - j * cpr;
    const int slot = hd + j < W ? hd + j : hd + j - W;
    const uint4 raw = *reinterpret_cast<const uint4*>(head_rows + (size_t)slot * cols + c * epc);
    float f[epc];
    unpack<TI>(raw, f);
    float4* d = reinterpret_cast<float4*>(dst + (size_t)j * cols + c * epc);
#pragma unroll
    for (int e = 0; e < epc / 4; ++e) d[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2], f[4 * e + 3]);
  }
}

constexpr int kDFoldThreads = 256;

// Rows of the fold held per thread, and lanes per row: each lane holds 16
// columns of each of its kFoldRowsPT rows (float4 chunks q, q + L, q + 2L and
// q + 3L of the row, L = DK / 16 lanes per row), so a thread runs four
// independent per-entry chains and the lanes of a row share every k_j load.
constexpr int kFoldRowsPT = 4;
template <int DK>
__host__ __device__ constexpr int fold_lanes_per_row() { return DK / 16; }

// The n-entry fold of a thread's kFoldRowsPT rows of one head, held in
// registers (rows r[i], present when i < nr; absent rows compute on a
// copy of row 0 and are never stored). Each row evolves independently,
//   s <- alpha (.) s;  s <- s + beta (v[r] - s . k) k   for j = 0..n-1,
// with the entries (float, entry order) in shared memory. A scalar GDN gate
// is applied lazily: the rows hold s / gam, gam the product of the gates so
// far, and are rescaled once at the end -- or as soon as gam drops below
// kGamFloor, which includes a gate of 0 (the rows are then reset to 0):
// the running inverse 1 / gam is never formed from a huge or infinite
// reciprocal. k_j (and a KDA gate row) are read
// once per entry from shared memory for all four rows: the L lanes of a row
// read L consecutive float4, one conflict-free broadcast per chunk.
constexpr float kGamFloor = 0x1p-32f;

template <int DK, bool KDA>
__device__ __forceinline__ void fold_rows(float2 (&s)[kFoldRowsPT][8], const int (&r)[kFoldRowsPT],
                                          int n, int DV, int q, const float* kbuf,
                                          const float* abuf, const float* vbuf,
                                          const float* bbuf, const float* rbuf) {
  constexpr int L = fold_lanes_per_row<DK>();
  float gam = 1.f, igam = 1.f;  // GDN: product of the gates so far, and its inverse
  for (int j = 0; j < n; ++j) {
    const float4* kj = reinterpret_cast<const float4*>(kbuf + (size_t)j * DK) + q;
    float4 kc[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) kc[m] = kj[L * m];
    if (KDA) {
      const float4* aj = reinterpret_cast<const float4*>(abuf + (size_t)j * DK) + q;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 u = aj[L * m];
        const float2 g0 = make_float2(u.x, u.y), g1 = make_float2(u.z, u.w);
#pragma unroll
        for (int i = 0; i < kFoldRowsPT; ++i) {
          s[i][2 * m] = __fmul2_rn(s[i][2 * m], g0);
          s[i][2 * m + 1] = __fmul2_rn(s[i][2 * m + 1], g1);
        }
      }
    } else {
      gam *= abuf[j];
      if (!(gam >= kGamFloor)) {  // the lazy product is applied to the rows now
        const float2 gg = make_float2(gam, gam);
#pragma unroll
        for (int i = 0; i < kFoldRowsPT; ++i) {
#pragma unroll
          for (int m = 0; m < 8; ++m) s[i][m] = __fmul2_rn(s[i][m], gg);
        }
        gam = 1.f;
        igam = 1.f;
      } else {
        igam *= rbuf[j];
      }
    }
    float dot[kFoldRowsPT];
#pragma unroll
    for (int i = 0; i < kFoldRowsPT; ++i) {  // two accumulators per row
      float2 d0 = make_float2(0.f, 0.f), d1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        d0 = __ffma2_rn(s[i][2 * m], make_float2(kc[m].x, kc[m].y), d0);
        d1 = __ffma2_rn(s[i][2 * m + 1], make_float2(kc[m].z, kc[m].w), d1);
      }
      dot[i] = (d0.x + d0.y) + (d1.x + d1.y);
    }
#pragma unroll
    for (int o = 1; o < L; o <<= 1) {
#pragma unroll
      for (int i = 0; i < kFoldRowsPT; ++i) dot[i] += __shfl_xor_sync(kFull, dot[i], o);
    }
    const float bj = bbuf[j];
    const float* vj = vbuf + (size_t)j * DV;
#pragma unroll
    for (int i = 0; i < kFoldRowsPT; ++i) {
      float c = KDA ? bj * (vj[r[i]] - dot[i]) : bj * (vj[r[i]] - dot[i] * gam) * igam;
      const float2 cc = make_float2(c, c);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        s[i][2 * m] = __ffma2_rn(cc, make_float2(kc[m].x, kc[m].y), s[i][2 * m]);
        s[i][2 * m + 1] = __ffma2_rn(cc, make_float2(kc[m].z, kc[m].w), s[i][2 * m + 1]);
      }
    }
  }
  if (!KDA) {
    const float2 gg = make_float2(gam, gam);
#pragma unroll
    for (int i = 0; i < kFoldRowsPT; ++i) {
#pragma unroll
      for (int m = 0; m < 8; ++m) s[i][m] = __fmul2_rn(s[i][m], gg);
    }
  }
}

// A thread's rows in the layout of fold_rows from a row-major [rows][DK]
// FP32 block (global or shared memory): row i is block row r[i].
template <int DK>
__device__ __forceinline__ void load_rows(const float* block, const int (&r)[kFoldRowsPT], int q,
                                          float2 (&s)[kFoldRowsPT][8]) {
  constexpr int L = fold_lanes_per_row<DK>();
#pragma unroll
  for (int i = 0; i < kFoldRowsPT; ++i) {
    const float4* p = reinterpret_cast<const float4*>(block + (size_t)r[i] * DK) + q;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float4 u = p[L * m];
      s[i][2 * m] = make_float2(u.x, u.y);
      s[i][2 * m + 1] = make_float2(u.z, u.w);
    }
  }
}

// The folded rows back to the FP32 checkpoint (row i is state row base + r[i],
// stored when i < nr) and, when Sr is set, to the BF16 read copy (round to
// nearest even).
template <int DK>
__device__ __forceinline__ void store_rows(float* S, bf16* Sr, size_t base, const int (&r)[kFoldRowsPT],
                                           int nr, int q, const float2 (&s)[kFoldRowsPT][8]) {
  constexpr int L = fold_lanes_per_row<DK>();
#pragma unroll
  for (int i = 0; i < kFoldRowsPT; ++i) {
    if (i >= nr) break;
    const size_t g = base + r[i];
    float4* row = reinterpret_cast<float4*>(S + g * DK) + q;
#pragma unroll
    for (int m = 0; m < 4; ++m)
      row[L * m] = make_float4(s[i][2 * m].x, s[i][2 * m].y, s[i][2 * m + 1].x, s[i][2 * m + 1].y);
    if (Sr) {
      uint2* rr = reinterpret_cast<uint2*>(Sr + g * DK) + q;
#pragma unroll
      for (int m = 0; m < 4; ++m)
        rr[L * m] = make_uint2(pack_bf16x2(s[i][2 * m].x, s[i][2 * m].y),
                               pack_bf16x2(s[i][2 * m + 1].x, s[i][2 * m + 1].y));
    }
  }
}

// The token of a fused step as the fold's output needs it, from one warp:
// u = A_t (scale q_t) into ubuf[DK], ce = scale beta_t (k_t . q_t) into *ce
// and v_t into vt[DV] (floats), from the token's q, k, v rows, its gate
// (a scalar, or a row for KDA) and beta. A_t x = alpha (.) (x - beta (k . x) k).
template <int DK, typename TI, bool KDA>
__device__ __forceinline__ void token_terms(const TI* q, const TI* k, const TI* v,
                                            const float* alpha, float bt, float scale, int DV,
                                            float* ubuf, float* vt, float* ce, int lane) {
  constexpr int E = DK / 32;
  float qf[E], kf[E];
  load_vec<TI, E>(q + lane * E, qf);
  load_vec<TI, E>(k + lane * E, kf);
  float kq = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) kq = fmaf(kf[e], qf[e], kq);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) kq += __shfl_xor_sync(kFull, kq, o);
  kq *= scale;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float al = KDA ? alpha[lane * E + e] : alpha[0];
    ubuf[lane * E + e] = al * (scale * qf[e] - bt * kq * kf[e]);
  }
  for (int r = lane; r < DV; r += 32) vt[r] = to_f(v[r]);
  if (lane == 0) *ce = bt * kq;
}

// The fold's rows times u: o[obase + r[i]] = S'_read[r[i]] . u + ce vt[r[i]]
// (i < nr), S'_read the rows as the read copy holds them (BF16-rounded when
// round16), reduced over the L lanes of a row.
template <int DK>
__device__ __forceinline__ void out_rows(float* o, size_t obase, const int (&r)[kFoldRowsPT], int nr,
                                         int q, const float2 (&s)[kFoldRowsPT][8], bool round16,
                                         const float* ubuf, const float* vt, float ce) {
  constexpr int L = fold_lanes_per_row<DK>();
  const float4* u4 = reinterpret_cast<const float4*>(ubuf) + q;
  float acc[kFoldRowsPT];
#pragma unroll
  for (int i = 0; i < kFoldRowsPT; ++i) {
    float sacc = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float4 u = u4[L * m];
      float x0 = s[i][2 * m].x, x1 = s[i][2 * m].y, x2 = s[i][2 * m + 1].x, x3 = s[i][2 * m + 1].y;
      if (round16) {
        const uint32_t p0 = pack_bf16x2(x0, x1), p1 = pack_bf16x2(x2, x3);
        x0 = bf16_lo(p0), x1 = bf16_hi(p0), x2 = bf16_lo(p1), x3 = bf16_hi(p1);
      }
      sacc = fmaf(x0, u.x, fmaf(x1, u.y, fmaf(x2, u.z, fmaf(x3, u.w, sacc))));
    }
    acc[i] = sacc;
  }
#pragma unroll
  for (int sh = 1; sh < L; sh <<= 1) {
#pragma unroll
    for (int i = 0; i < kFoldRowsPT; ++i) acc[i] += __shfl_xor_sync(kFull, acc[i], sh);
  }
  if (q == 0) {
#pragma unroll
    for (int i = 0; i < kFoldRowsPT; ++i)
      if (i < nr) o[obase + r[i]] = fmaf(ce, vt[r[i]], acc[i]);
  }
}

// The token of a fused step into ring slot `slot` of head t (block threads):
// q (when stored), k, v, the gate and beta.
template <int DK, typename TI, bool KDA>
__device__ __forceinline__ void append_token(const DFold& a, size_t t, int slot, int W, int DV) {
  const int Wd = ring_wd(W);
  constexpr int kv = 16 / (int)sizeof(TI);  // elements per 16-byte copy
  const size_t kr = (t * W + slot) * DK, vr = (t * W + slot) * (size_t)DV;
  for (int c = threadIdx.x; c < DK / kv; c += blockDim.x) {
    reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.ring_kw) + kr)[c] =
        reinterpret_cast<const uint4*>(reinterpret_cast<const TI*>(a.k) + t * DK)[c];
    if (a.ring_q)
      reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.ring_q) + kr)[c] =
          reinterpret_cast<const uint4*>(reinterpret_cast<const TI*>(a.q) + t * DK)[c];
  }
  for (int c = threadIdx.x; c < DV / kv; c += blockDim.x)
    reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.ring_vw) + vr)[c] =
        reinterpret_cast<const uint4*>(reinterpret_cast<const TI*>(a.v) + t * DV)[c];
  if (KDA) {
    for (int c = threadIdx.x; c < DK; c += blockDim.x)
      a.ring_alphaw[(t * W + slot) * DK + c] = a.alpha[t * DK + c];
  } else if (threadIdx.x == 0) {
    a.ring_alphaw[t * Wd + slot] = a.alpha[t];
  }
  if (threadIdx.x == 0) a.ring_betaw[t * Wd + slot] = a.beta[t];
}

// Consolidate for the delta-rule layers, synchronous form: one block per
// folding head (a parallel pre-scan of the pointers lists them). The head's
// n entries (k, v, gates, beta) are staged as float, then each thread folds
// four rows x 16 columns in registers (fold_rows). Rows are read
// once and written once (FP32 checkpoint and BF16 read copy). Used where the
// prefetching form below does not fit two blocks per SM.
template <int DK, typename TI, bool KDA>
__global__ void __launch_bounds__(kDFoldThreads, 2) delta_fold_kernel(const DFold a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ FoldList fl;
  constexpr int LPR = fold_lanes_per_row<DK>();  // lanes per row
  constexpr int SLOTS = kDFoldThreads / LPR;      // row slots per pass
  const int tid = threadIdx.x, q = tid % LPR, rs = tid / LPR;
  const int H = a.H, DV = a.DV, W = a.W, Wd = ring_wd(W);
  float* kbuf = reinterpret_cast<float*>(smem);                   // [W][DK]
  float* abuf = kbuf + (size_t)W * DK;                            // KDA [W][DK], GDN [W]
  float* vbuf = abuf + align_up((size_t)W * (KDA ? DK : 1), 4);   // [W][DV]
  float* bbuf = vbuf + (size_t)W * DV;                            // [W]
  float* rbuf = bbuf + W;                                         // GDN [W]: 1 / alpha_j
  float* ubuf = kbuf + align_up((size_t)(rbuf - kbuf) + W, 4);    // fused step: u [DK],
  float* vt = ubuf + DK;                                          // v_t [DV], ce
  float* cep = vt + DV;
  const TI* rk = reinterpret_cast<const TI*>(a.ring_k);
  const TI* rv = reinterpret_cast<const TI*>(a.ring_v);

  griddep_wait();  // a fused step's decode grid has written the flags and pointers
  collect_folds(fl, (long long)a.batch * H, H, a.len, a.head, a.status, W, a.k_next, a.force,
                a.flags);
  for (int f = 0; f < fl.count; ++f) {
    const int t = fl.tile[f], n = fl.len[f], hd = fl.head[f];
    const int seq = t / H;
    stage_rows_f32<TI>(kbuf, rk + (size_t)t * W * DK, DK, n, hd, W);
    stage_rows_f32<TI>(vbuf, rv + (size_t)t * W * DV, DV, n, hd, W);
    if (KDA) stage_rows_f32<float>(abuf, a.ring_alpha + (size_t)t * W * DK, DK, n, hd, W);
    for (int j = tid; j < n; j += kDFoldThreads) {
      const int slot = hd + j < W ? hd + j : hd + j - W;
      bbuf[j] = a.ring_beta[(size_t)t * Wd + slot];
      if (!KDA) {
        const float al = a.ring_alpha[(size_t)t * Wd + slot];
        abuf[j] = al;
        rbuf[j] = 1.f / al;
      }
    }
    if (a.flags && tid < 32)
      token_terms<DK, TI, KDA>(reinterpret_cast<const TI*>(a.q) + (size_t)t * DK,
                               reinterpret_cast<const TI*>(a.k) + (size_t)t * DK,
                               reinterpret_cast<const TI*>(a.v) + (size_t)t * DV,
                               a.alpha + (KDA ? (size_t)t * DK : (size_t)t), a.beta[t], a.scale,
                               DV, ubuf, vt, cep, tid);
    __syncthreads();
    for (int r0 = rs; r0 < DV; r0 += kFoldRowsPT * SLOTS) {
      // rows r0 + i * SLOTS; DV is a multiple of 32, so nr is uniform over a warp
      int r[kFoldRowsPT], nr = 0;
#pragma unroll
      for (int i = 0; i < kFoldRowsPT; ++i) {
        const int ri = r0 + i * SLOTS;
        nr += ri < DV;
        r[i] = ri < DV ? ri : r0;
      }
      float2 sv[kFoldRowsPT][8];
      load_rows<DK>(a.S + (size_t)t * DV * DK, r, q, sv);
      fold_rows<DK, KDA>(sv, r, n, DV, q, kbuf, abuf, vbuf, bbuf, rbuf);
      store_rows<DK>(a.S, a.Sr, (size_t)t * DV, r, nr, q, sv);
      if (a.flags) out_rows<DK>(a.o, (size_t)t * DV, r, nr, q, sv, a.Sr != nullptr, ubuf, vt, *cep);
    }
    // fused step: the token into entry 0's old slot, now that every entry is read
    if (a.flags) append_token<DK, TI, KDA>(a, (size_t)t, (hd + n) % W, W, DV);
    __syncthreads();
    if (tid == 0)
      arrive_and_finish(a.sync + seq, 1, H, [&] {
        a.head[seq] = (hd + n) % W;
        a.len[seq] = a.flags ? 1 : 0;
      });
  }
}

// Rows of the prefetching fold: one row chunk of a head per unit, the rows
// that one pass of the block's threads holds (kFoldRowsPT per row slot).
__host__ __device__ constexpr int fold_chunk_rows(int DK, int DV) {
  return DV < kFoldRowsPT * kDFoldThreads * 16 / DK ? DV : kFoldRowsPT * kDFoldThreads * 16 / DK;
}

__host__ __device__ inline size_t smem_take(size_t& o, size_t bytes) {
  const size_t at = o;
  o = align_up(o + bytes, 128);
  return at;
}

// Shared-memory layout of the prefetching fold (byte offsets): the staged
// row chunk of S; the next unit's raw ring entries (k, v, KDA gate rows in
// entry order; the scalar fields' whole [Wd] blocks in slot order); the
// current unit's entries widened to float; one mbarrier.
struct DFoldSmem {
  size_t s, kraw, vraw, araw, braw, kbuf, abuf, vbuf, bbuf, rbuf, ubuf, vt, ce, tq, tk, tv, ta, tb,
      bar, total;
  __host__ __device__ DFoldSmem(int DK, int DV, int W, int ti, bool kda) {
    const size_t R = fold_chunk_rows(DK, DV), Wd = ring_wd(W);
    size_t o = 0;
    s = smem_take(o, R * DK * 4);
    kraw = smem_take(o, (size_t)W * DK * ti);
    vraw = smem_take(o, (size_t)W * DV * ti);
    araw = smem_take(o, kda ? (size_t)W * DK * 4 : Wd * 4);
    braw = smem_take(o, Wd * 4);
    kbuf = smem_take(o, (size_t)W * DK * 4);
    abuf = smem_take(o, kda ? (size_t)W * DK * 4 : (size_t)W * 4);
    vbuf = smem_take(o, (size_t)W * DV * 4);
    bbuf = smem_take(o, (size_t)W * 4);
    rbuf = smem_take(o, (size_t)W * 4);
    ubuf = smem_take(o, (size_t)DK * 4);  // fused step: u, v_t and ce of the token,
    vt = smem_take(o, (size_t)DV * 4);    // and the next unit's token as it arrives
    ce = smem_take(o, 16);
    tq = smem_take(o, (size_t)DK * ti);
    tk = smem_take(o, (size_t)DK * ti);
    tv = smem_take(o, (size_t)DV * ti);
    ta = smem_take(o, kda ? (size_t)DK * 4 : 16);
    tb = smem_take(o, 16);
    bar = smem_take(o, 8);
    total = o;
  }
};

// Ring rows of `cols` elements of entries 0..n-1 of one head (entry j in
// slot (hd + j) mod W of the head's [W][cols] block) into dst [n][cols] with
// 16-byte cp.async from every thread (cols * sizeof(T) a multiple of 16).
template <typename T>
__device__ __forceinline__ void prefetch_ring_rows(T* dst, const T* head_rows, int cols, int n,
                                                   int hd, int W) {
  constexpr int epc = 16 / (int)sizeof(T);
  const int cpr = cols / epc;
  for (int idx = threadIdx.x; idx < n * cpr; idx += blockDim.x) {
    const int j = idx / cpr, c = idx - j * cpr;
    const int slot = hd + j < W ? hd + j : hd + j - W;
    cp_async16(dst + (size_t)j * cols + c * epc, head_rows + (size_t)slot * cols + c * epc);
  }
}

// `count` elements (a multiple of 16 bytes' worth) of shared memory widened to float.
template <typename T>
__device__ __forceinline__ void widen_smem(float* dst, const T* src, int count) {
  constexpr int epc = 16 / (int)sizeof(T);
  for (int idx = threadIdx.x; idx < count / epc; idx += blockDim.x) {
    float f[epc];
    unpack<T>(reinterpret_cast<const uint4*>(src)[idx], f);
    float4* d = reinterpret_cast<float4*>(dst + (size_t)idx * epc);
#pragma unroll
    for (int e = 0; e < epc / 4; ++e) d[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2], f[4 * e + 3]);
  }
}

// Consolidate for the delta-rule layers, prefetching form. The same fold as
// delta_fold_kernel on units of (folding head, row chunk), but the next
// unit's row chunk (one bulk copy, completion on an mbarrier) and ring
// entries (cp.async) are in flight while the block folds the current one, so
// the state stream overlaps the serial per-entry arithmetic. Per unit:
// wait for its copies; widen its entries to float; move its rows from shared
// memory to registers; barrier; issue the next unit's copies; fold and store.
// Each unit's arrival on the sequence's counter comes after the barrier that
// follows its stores; the last of the H x chunks arrivals moves the pointers.
template <int DK, typename TI, bool KDA>
__global__ void __launch_bounds__(kDFoldThreads, 2) delta_fold_stream_kernel(const DFold a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ FoldList fl;
  constexpr int LPR = fold_lanes_per_row<DK>();  // lanes per row
  constexpr int SLOTS = kDFoldThreads / LPR;      // row slots per pass
  const int tid = threadIdx.x, q = tid % LPR, rs = tid / LPR;
  const int H = a.H, DV = a.DV, W = a.W, Wd = ring_wd(W);
  const int R = fold_chunk_rows(DK, DV), nch = (DV + R - 1) / R;
  const DFoldSmem L(DK, DV, W, (int)sizeof(TI), KDA);
  float* sS = reinterpret_cast<float*>(smem + L.s);
  TI* kraw = reinterpret_cast<TI*>(smem + L.kraw);
  TI* vraw = reinterpret_cast<TI*>(smem + L.vraw);
  float* araw = reinterpret_cast<float*>(smem + L.araw);
  float* braw = reinterpret_cast<float*>(smem + L.braw);
  float* kbuf = reinterpret_cast<float*>(smem + L.kbuf);
  float* abuf = reinterpret_cast<float*>(smem + L.abuf);
  float* vbuf = reinterpret_cast<float*>(smem + L.vbuf);
  float* bbuf = reinterpret_cast<float*>(smem + L.bbuf);
  float* rbuf = reinterpret_cast<float*>(smem + L.rbuf);
  float* ubuf = reinterpret_cast<float*>(smem + L.ubuf);
  float* vt = reinterpret_cast<float*>(smem + L.vt);
  float* cep = reinterpret_cast<float*>(smem + L.ce);
  TI* tq = reinterpret_cast<TI*>(smem + L.tq);  // the fused step's token (raw)
  TI* tk = reinterpret_cast<TI*>(smem + L.tk);
  TI* tv = reinterpret_cast<TI*>(smem + L.tv);
  float* ta = reinterpret_cast<float*>(smem + L.ta);
  float* tb = reinterpret_cast<float*>(smem + L.tb);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
  const TI* rk = reinterpret_cast<const TI*>(a.ring_k);
  const TI* rv = reinterpret_cast<const TI*>(a.ring_v);
  const uint64_t pol = l2_evict_first_policy();
  constexpr int kTV = 16 / (int)sizeof(TI);  // elements per 16-byte copy

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  griddep_wait();  // a fused step's decode grid has written the flags and pointers
  // (its barriers also publish the mbarrier's initialisation)
  collect_folds(fl, (long long)a.batch * H, H, a.len, a.head, a.status, W, a.k_next, a.force,
                a.flags);
  const int units = fl.count * nch;

  auto issue = [&](int u) {
    const int f = u / nch, c0 = (u - f * nch) * R;
    const int t = fl.tile[f], n = fl.len[f], hd = fl.head[f];
    const int rows = DV - c0 < R ? DV - c0 : R;
    if (tid == 0) {
      const uint32_t bytes = (uint32_t)rows * DK * 4;
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(sS, a.S + ((size_t)t * DV + c0) * DK, bytes, bar, pol);
    }
    prefetch_ring_rows<TI>(kraw, rk + (size_t)t * W * DK, DK, n, hd, W);
    prefetch_ring_rows<TI>(vraw, rv + (size_t)t * W * DV, DV, n, hd, W);
    if (KDA) prefetch_ring_rows<float>(araw, a.ring_alpha + (size_t)t * W * DK, DK, n, hd, W);
    for (int i = tid; i < Wd / 4; i += kDFoldThreads) {
      cp_async16(braw + 4 * i, a.ring_beta + (size_t)t * Wd + 4 * i);
      if (!KDA) cp_async16(araw + 4 * i, a.ring_alpha + (size_t)t * Wd + 4 * i);
    }
    if (a.flags) {  // the fused step's token of head t
      const TI* qg = reinterpret_cast<const TI*>(a.q) + (size_t)t * DK;
      const TI* kg = reinterpret_cast<const TI*>(a.k) + (size_t)t * DK;
      const TI* vg = reinterpret_cast<const TI*>(a.v) + (size_t)t * DV;
      for (int i = tid; i < DK / kTV; i += kDFoldThreads) {
        cp_async16(tq + i * kTV, qg + i * kTV);
        cp_async16(tk + i * kTV, kg + i * kTV);
      }
      for (int i = tid; i < DV / kTV; i += kDFoldThreads) cp_async16(tv + i * kTV, vg + i * kTV);
      if (KDA) {
        for (int i = tid; i < DK / 4; i += kDFoldThreads)
          cp_async16(ta + 4 * i, a.alpha + (size_t)t * DK + 4 * i);
      } else if (tid == 0) {
        cp_async4(ta, a.alpha + t);
      }
      if (tid == 0) cp_async4(tb, a.beta + t);
    }
    cp_async_commit();
  };
  // The last arrival of a sequence's units moves its pointers. Thread 0
  // arrives for a unit after the barrier that follows the unit's stores, and
  // looks at the count it got back one unit later, so the atomic's round trip
  // is off the block's path. No fence before it: the pointers it moves are
  // read in this kernel only by the blocks that fold that sequence, before
  // their own arrivals, and the state rows only by later launches.
  int pend_seq = -1, pend_old = 0, pend_head = 0;
  auto settle = [&]() {
    if (pend_seq >= 0 && pend_old + 1 == H * nch) {
      a.head[pend_seq] = pend_head;
      a.len[pend_seq] = a.flags ? 1 : 0;
      a.sync[pend_seq] = 0;
    }
    pend_seq = -1;
  };
  auto arrive = [&](int u) {
    settle();
    const int f = u / nch;
    pend_seq = fl.tile[f] / H;
    pend_head = (fl.head[f] + fl.len[f]) % W;
    pend_old = atomicAdd(a.sync + pend_seq, 1);
  };

  if (units > 0) issue(0);
  uint32_t ph = 0;
  for (int u = 0; u < units; ++u) {
    const int f = u / nch, c0 = (u - f * nch) * R;
    const int t = fl.tile[f], n = fl.len[f], hd = fl.head[f];
    const int rows = DV - c0 < R ? DV - c0 : R;
    cp_async_wait_all();
    const bool landed = mbar_wait(bar, ph);
    // unit u's copies are visible to every thread, and every thread is done
    // with unit u - 1 (its float entries, its stores)
    const bool ok = __syncthreads_and(landed) != 0;
    if (tid == 0 && u > 0) arrive(u - 1);
    if (!ok) {
      if (tid == 0) {
        settle();
        for (int g = f; g < fl.count; ++g) atomicOr(a.status + fl.tile[g] / H, REPLAYSSM_SEQ_TIMEOUT);
        mbar_wait(bar, ph);  // no bulk copy may land after the block exits
      }
      return;
    }
    ph ^= 1;
    widen_smem<TI>(kbuf, kraw, n * DK);
    widen_smem<TI>(vbuf, vraw, n * DV);
    if (KDA) widen_smem<float>(abuf, araw, n * DK);
    for (int j = tid; j < n; j += kDFoldThreads) {
      const int slot = hd + j < W ? hd + j : hd + j - W;
      bbuf[j] = braw[slot];
      if (!KDA) {
        const float al = araw[slot];
        abuf[j] = al;
        rbuf[j] = 1.f / al;
      }
    }
    // chunk rows rs + i * SLOTS; rows is a multiple of 32, so nr is uniform
    // over each warp
    int r[kFoldRowsPT], nr = 0;
#pragma unroll
    for (int i = 0; i < kFoldRowsPT; ++i) {
      const int ri = rs + i * SLOTS;
      nr += ri < rows;
      r[i] = ri < rows ? ri : rs;
    }
    float2 sv[kFoldRowsPT][8];
    if (nr > 0) load_rows<DK>(sS, r, q, sv);
    if (a.flags) {
      if (tid < 32)
        token_terms<DK, TI, KDA>(tq, tk, tv, ta, tb[0], a.scale, DV, ubuf, vt, cep, tid);
      // after the head's last chunk has landed (every entry of the head
      // staged) the token goes into entry 0's old slot
      if (c0 + rows == DV) {
        const int slot = (hd + n) % W;
        const size_t kr = ((size_t)t * W + slot) * DK, vr = ((size_t)t * W + slot) * DV;
        for (int i = tid; i < DK / kTV; i += kDFoldThreads) {
          reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.ring_kw) + kr)[i] = reinterpret_cast<const uint4*>(tk)[i];
          if (a.ring_q)
            reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.ring_q) + kr)[i] = reinterpret_cast<const uint4*>(tq)[i];
        }
        for (int i = tid; i < DV / kTV; i += kDFoldThreads)
          reinterpret_cast<uint4*>(reinterpret_cast<TI*>(a.ring_vw) + vr)[i] = reinterpret_cast<const uint4*>(tv)[i];
        if (KDA) {
          for (int i = tid; i < DK; i += kDFoldThreads) a.ring_alphaw[((size_t)t * W + slot) * DK + i] = ta[i];
        } else if (tid == 0) {
          a.ring_alphaw[(size_t)t * Wd + slot] = ta[0];
        }
        if (tid == 0) a.ring_betaw[(size_t)t * Wd + slot] = tb[0];
      }
    }
    __syncthreads();  // entries widened; the staged chunk and raw entries are free
    if (u + 1 < units) issue(u + 1);
    if (nr > 0) {
      int rg[kFoldRowsPT];  // rows within the head
#pragma unroll
      for (int i = 0; i < kFoldRowsPT; ++i) rg[i] = c0 + r[i];
      fold_rows<DK, KDA>(sv, rg, n, DV, q, kbuf, abuf, vbuf, bbuf, rbuf);
      store_rows<DK>(a.S, a.Sr, (size_t)t * DV, rg, nr, q, sv);
      if (a.flags) out_rows<DK>(a.o, (size_t)t * DV, rg, nr, q, sv, a.Sr != nullptr, ubuf, vt, *cep);
    }
  }
  if (units > 0) {
    __syncthreads();
    if (tid == 0) {
      arrive(units - 1);
      settle();
    }
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

struct DConvSpec {
  int batch, H, DV, K;
  const float* S;       // [b, H, DV, DK], not modified
  const void* q;        // drafts [b, K, H, ...]
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  float scale;
  float* snap;          // [b, K, H, DV, DK]: the state after drafts 0..i
  float* o;             // [b, K, H, DV]
};

// Conventional speculative verify, the baseline the pointer method replaces:
// the recurrence runs through the K drafts in order and the state after each
// draft is written out as a snapshot (from which accept restores the state
// of the accepted prefix). Same row layout as the conventional step: one warp
// per 8 rows of one head, 8 lanes per row; the rows stay in registers across
// the drafts.
template <int DK, typename TI, bool KDA>
__global__ void __launch_bounds__(kThreads) delta_conventional_verify_kernel(const DConvSpec a) {
  constexpr int CH = DK / 32;  // float4 chunks per lane
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int groups = a.DV / 8, H = a.H, K = a.K;
  if (gw >= (long long)a.batch * H * groups) return;
  const long long t = gw / groups;  // seq * H + h
  const long long seq = t / H, h = t - seq * H;
  const int r0 = (int)(gw - t * groups) * 8;
  const int sub = lane >> 3, c8 = lane & 7;
  float4 sv[2][CH];
#pragma unroll
  for (int st = 0; st < 2; ++st) {
    const float4* row = reinterpret_cast<const float4*>(a.S + (t * a.DV + r0 + st * 4 + sub) * DK);
#pragma unroll
    for (int m = 0; m < CH; ++m) sv[st][m] = row[c8 + 8 * m];
  }
  for (int i = 0; i < K; ++i) {
    const long long ti = (seq * K + i) * H + h;  // draft i of this head
    const TI* qi = reinterpret_cast<const TI*>(a.q) + ti * DK;
    const TI* ki = reinterpret_cast<const TI*>(a.k) + ti * DK;
    const TI* vi = reinterpret_cast<const TI*>(a.v) + ti * a.DV;
    float kq[CH][4], qq[CH][4], al[CH][4];
    float kqdot = 0.f;
#pragma unroll
    for (int m = 0; m < CH; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = (c8 + 8 * m) * 4 + e;
        kq[m][e] = to_f(ki[c]);
        qq[m][e] = to_f(qi[c]);
        al[m][e] = KDA ? a.alpha[ti * DK + c] : a.alpha[ti];
        kqdot = fmaf(kq[m][e], qq[m][e], kqdot);
      }
    kqdot += __shfl_xor_sync(kFull, kqdot, 1);
    kqdot += __shfl_xor_sync(kFull, kqdot, 2);
    kqdot += __shfl_xor_sync(kFull, kqdot, 4);
    const float be = a.beta[ti];
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      const int r = r0 + st * 4 + sub;
      float d1 = 0.f, d2 = 0.f;
#pragma unroll
      for (int m = 0; m < CH; ++m) {
        sv[st][m].x *= al[m][0];
        sv[st][m].y *= al[m][1];
        sv[st][m].z *= al[m][2];
        sv[st][m].w *= al[m][3];
        d1 = fmaf(sv[st][m].x, kq[m][0], d1);
        d1 = fmaf(sv[st][m].y, kq[m][1], d1);
        d1 = fmaf(sv[st][m].z, kq[m][2], d1);
        d1 = fmaf(sv[st][m].w, kq[m][3], d1);
        d2 = fmaf(sv[st][m].x, qq[m][0], d2);
        d2 = fmaf(sv[st][m].y, qq[m][1], d2);
        d2 = fmaf(sv[st][m].z, qq[m][2], d2);
        d2 = fmaf(sv[st][m].w, qq[m][3], d2);
      }
#pragma unroll
      for (int o = 1; o <= 4; o <<= 1) {
        d1 += __shfl_xor_sync(kFull, d1, o);
        d2 += __shfl_xor_sync(kFull, d2, o);
      }
      const float c = be * (to_f(vi[r]) - d1);
      float4* snap = reinterpret_cast<float4*>(a.snap + (ti * a.DV + r) * DK);
#pragma unroll
      for (int m = 0; m < CH; ++m) {
        sv[st][m] = make_float4(fmaf(c, kq[m][0], sv[st][m].x), fmaf(c, kq[m][1], sv[st][m].y),
                                fmaf(c, kq[m][2], sv[st][m].z), fmaf(c, kq[m][3], sv[st][m].w));
        snap[c8 + 8 * m] = sv[st][m];
      }
      if (c8 == 0) a.o[ti * a.DV + r] = a.scale * fmaf(c, kqdot, d2);
    }
  }
}

#include "delta_gram.cuh"

// cuTensorMapEncodeTiled from the CUDA driver API, looked up once (null if absent).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// The tensor-core kernel serves speculative verify (K > 1) of GDN with a
// BF16 read copy and BF16 inputs, d_k of 64 or 128, d_v a multiple of 64 and
// windows up to kGramN entries; REPLAYSSM_DELTA_TENSOR_CORES=0 selects the
// FFMA kernel instead. (A decode has one query: S [q | k]^T is then about 16
// multiply-adds per state element on the mma.sync pipe against one FFMA per
// element, and the FFMA kernel is as fast: 61 us against 63 us per b256 call.)
bool gram_eligible(const replayssm_dims& d, const replayssm_state& s, int K) {
  if (K < 2 || d.kind != REPLAYSSM_GDN || !s.S_read || d.in_dtype != REPLAYSSM_BF16) return false;
  if ((d.dk != 64 && d.dk != 128) || d.dv % kGRows != 0 || d.window > kGramN || K > kGramQ) return false;
  if ((reinterpret_cast<uintptr_t>(s.S_read) & 15) != 0) return false;
  const char* e = std::getenv("REPLAYSSM_DELTA_TENSOR_CORES");
  return !(e && e[0] == '0');
}

// Prep warps and stages of the tensor-core kernel: among (NP, depth) with
// NP x depth x (units per head) a multiple of the consumer groups (each
// group then sees every fill of the prep stages it reads, so no parity wait
// can take an older phase) and at least 4 state stages, the most heads in
// flight (NP x depth), ties to more stages. (b512 K = 4 verify, measured
// before the prep stages held the value terms: 7 x 2 with 4 stages 205 us,
// 6 x 2 213 us, 6 x 1 with 8 stages 215 us. With them 7 x 2 needs 244 KB at
// d_k = d_v = 128 and 6 x 2 is the one that fits.)
struct GramConfig {
  int NS, NP, depth;
  size_t smem;
};
GramConfig gram_config(int DK, int DV, int W, int K, size_t optin) {
  GramConfig best{0, 0, 0, 0};
  const int nrb = DV / kGRows;
  const int cands[][2] = {{7, 2}, {6, 2}, {4, 3}, {4, 2}, {2, 4}, {6, 1}, {3, 2}, {2, 2}, {4, 1}, {2, 1}};
  for (const auto& c : cands) {
    const int NP = c[0], depth = c[1];
    if ((NP * depth * nrb) % kGGroups != 0) continue;
    const GSmem L0(DK, DV, W, K, 0, NP, depth);
    const size_t fixed = L0.total + 2048;  // + the block's static shared memory
    if (fixed >= optin) continue;
    const int NS = std::min((int)((optin - fixed) / (L0.stage + 16)), 12) / kGGroups * kGGroups;
    if (NS < 4) continue;
    const bool better = NP * depth > best.NP * best.depth || (NP * depth == best.NP * best.depth && NS > best.NS);
    if (better) best = GramConfig{NS, NP, depth, GSmem(DK, DV, W, K, NS, NP, depth).total};
  }
  return best;
}

template <int DK, int KMAX>
cudaError_t launch_gram(const DFused& f, const bf16* S, cudaStream_t st, bool& launched) {
  launched = false;
  const DeviceInfo& dev = device_info();
  const GramConfig c = gram_config(DK, f.DV, f.W, f.K, (size_t)dev.smem_optin);
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (c.NP == 0 || !encode) return cudaSuccess;  // not launched: the caller falls back
  DGram g;
  const cuuint64_t dims[2] = {(cuuint64_t)DK, (cuuint64_t)f.batch * f.H * f.DV};
  const cuuint64_t strides[1] = {(cuuint64_t)DK * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kGRows};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&g.tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16*>(S), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaSuccess;
  g.f = f;
  g.f.RB = kGRows;
  g.f.nrb = f.DV / kGRows;
  g.f.NS = c.NS;
  g.f.NP = c.NP;
  g.f.depth = c.depth;
  auto kern = delta_gram_kernel<DK, KMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem);
  if (e != cudaSuccess) return e;
  const long long heads = (long long)f.batch * f.H;
  const int grid = (int)std::min<long long>(heads, dev.sms);
  kern<<<grid, 32 * (2 * kGGroups + 1 + c.NP), c.smem, st>>>(g);
  launched = true;
  return cudaGetLastError();
}

// State rows per unit: about 16 KB (at least 32 rows, dividing DV).
int fused_rows(int DK, int ts, int DV) {
  int RB = std::max(32, 16384 / (DK * ts) / 32 * 32);
  RB = std::min(RB, DV);
  while (DV % RB) RB -= 32;
  return RB;
}

// Fused-kernel configuration: state stages, vector slots, prep warps and
// their pipeline depth. Among the settings that fit in shared memory with at
// least min_stages state stages, the one with most heads in flight in the
// prep warps (NP x depth) wins; ties go to depth 2, then to more stages.
struct FusedConfig {
  int NS, NSL, NP, depth;
  size_t smem;
};
// Fewest state stages a configuration may have: BF16 tiles stream fine from 4
// (more prep warps pay off there), FP32 tiles need 8.
constexpr int min_stages(int ts) { return ts == 2 ? 4 : 8; }

// Vector slots for NP prep warps: at least NP + 4, a multiple of NP, and
// with NSL x nrb a multiple of the consumer groups; 0 if no count up to
// kFMaxSlots has both. Prep warp w takes heads w, w + NP, ..., so with NP
// dividing NSL every fill of a slot comes from the same warp, in order.
// Consumer group g takes the heads whose units fall on it (unit = head x nrb
// + row block), so with NSL x nrb a multiple of the groups its heads repeat
// every NSL heads and it consumes every fill of each slot it uses. Neither
// side then waits on a slot whose previous fill it has not seen, so a parity
// wait can never take an older phase for the one it wants.
int vector_slots(int NP, int nrb) {
  auto gcd = [](int x, int y) {
    while (y) {
      const int t = x % y;
      x = y;
      y = t;
    }
    return x;
  };
  const int m = kFGroups / gcd(nrb, kFGroups);
  const int step = NP / gcd(NP, m) * m;  // lcm(NP, m)
  const int nsl = (NP + 4 + step - 1) / step * step;
  return nsl <= kFMaxSlots ? nsl : 0;
}

FusedConfig fused_config(int RB, int DK, int DV, int W, int K, int GU, bool kda, int ts, int ti,
                         size_t optin) {
  FusedConfig best{0, 0, 0, 0, 0};
  const int np_max = kFWarps - 1 - kFGroups * GU;
  for (int depth = 2; depth >= 1; --depth) {
    for (int NP = np_max; NP >= 1; --NP) {
      const int NSL = vector_slots(NP, DV / RB);
      if (NSL == 0) continue;
      const DFusedSmem L0(RB, DK, DV, W, K, 0, NSL, NP, depth, kda, ts, ti);
      const size_t fixed = L0.total + 1024;
      if (fixed >= optin) continue;
      const int fit = (int)((optin - fixed) / (L0.stage + 16));
      const int NS = std::min(fit, 12) / kFGroups * kFGroups;
      if (NS < min_stages(ts)) continue;
      const bool better = NP * depth > best.NP * best.depth ||
                          (NP * depth == best.NP * best.depth && NS > best.NS);
      if (better) {
        const DFusedSmem L(RB, DK, DV, W, K, NS, NSL, NP, depth, kda, ts, ti);
        best = FusedConfig{NS, NSL, NP, depth, L.total};
      }
      break;  // fewer warps at this depth only lowers NP * depth
    }
  }
  if (best.NP == 0) {  // tight: the fewest stages that still run
    const int NSL = vector_slots(1, DV / RB);
    const DFusedSmem L0(RB, DK, DV, W, K, 0, NSL, 1, 1, kda, ts, ti);
    const size_t fixed = L0.total + 1024;
    if (fixed < optin) {
      const int NS = std::min((int)((optin - fixed) / (L0.stage + 16)), 12) / kFGroups * kFGroups;
      if (NS >= kFGroups) {
        const DFusedSmem L(RB, DK, DV, W, K, NS, NSL, 1, 1, kda, ts, ti);
        best = FusedConfig{NS, NSL, 1, 1, L.total};
      }
    }
  }
  return best;
}

// Decode (K = 1) from the BF16 read copy. A configuration scores its prep
// warps plus its consumer warps per group (GU): a second consumer warp per
// group counts as much as a prep warp, and ties go to GU = 2, then to more
// state stages, then to depth 1. The prep warps' sweeps set the pace, but a
// consumer group also holds its stages while it computes; with KDA's larger
// prep stages only four state stages fit (one per group), and halving the
// group's time per unit is what keeps the stream going. Measured per call on
// the b256 layers: KDA 7 prep warps at GU = 2 70-73 us against 80 us with 8
// at GU = 1 (101 against 108 us per fused step); GDN 59.3 us either way (8
// stages); GDN 9 prep warps at GU = 1 61.3 us against 60.8 us with 8, and 10
// or 11 leave room for only 4 stages, 74 us. Zero NP: nothing fits.
FusedConfig decode_config(int RB, int DK, int DV, int W, bool kda, int ti, size_t optin, int& GU) {
  FusedConfig best{0, 0, 0, 0, 0};
  int best_gu = 0;
  const int gu_first = RB % 64 == 0 ? 2 : 1;
  for (int gu = gu_first; gu >= 1; --gu) {
    if (RB / gu > 128) continue;
    for (int depth = 1; depth <= 2; ++depth) {
      for (int NP = kFWarps - 1 - kFGroups * gu; NP >= 1; --NP) {
        const int NSL = vector_slots(NP, DV / RB);
        if (NSL == 0) continue;
        const DFusedSmem L0(RB, DK, DV, W, 1, 0, NSL, NP, depth, kda, 2, ti);
        const size_t fixed = L0.total + 1024;
        if (fixed >= optin) continue;
        const int NS = std::min((int)((optin - fixed) / (L0.stage + 16)), 12) / kFGroups * kFGroups;
        if (NS < min_stages(2)) continue;
        const int score = NP + gu, best_score = best.NP + best_gu;
        const bool better =
            score > best_score ||
            (score == best_score && gu == best_gu &&
             (NS > best.NS || (NS == best.NS && depth < best.depth)));
        if (better) {
          best = FusedConfig{NS, NSL, NP, depth, DFusedSmem(RB, DK, DV, W, 1, NS, NSL, NP, depth, kda, 2, ti).total};
          best_gu = gu;
        }
        break;  // fewer prep warps at this depth only lose
      }
    }
  }
  if (best.NP > 0) GU = best_gu;
  return best;
}

// Tile shape, stage count and template instance of the fused kernel.
template <int DK, typename TS, typename TI, bool KDA, int KMAX>
cudaError_t launch_fused(DFused a, cudaStream_t st) {
  const DeviceInfo& dev = device_info();
  const int RB = fused_rows(DK, sizeof(TS), a.DV);
  a.RB = RB;
  a.nrb = a.DV / RB;
  a.GU = RB % 64 == 0 ? 2 : 1;  // each warp's share must be whole 32-row groups
  if (RB / a.GU > 128 || a.K > KMAX) return cudaErrorInvalidValue;
  FusedConfig c{0, 0, 0, 0, 0};
  if (a.K == 1 && sizeof(TS) == 2)
    c = decode_config(RB, DK, a.DV, a.W, KDA, sizeof(TI), (size_t)dev.smem_optin, a.GU);
  if (c.NP == 0)
    c = fused_config(RB, DK, a.DV, a.W, a.K, a.GU, KDA, sizeof(TS), sizeof(TI), (size_t)dev.smem_optin);
  if (c.NP == 0) return cudaErrorInvalidConfiguration;
  a.NS = c.NS;
  a.NSL = c.NSL;
  a.NP = c.NP;
  a.depth = c.depth;
  auto kern = delta_fused_kernel<DK, TS, TI, KDA, KMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem);
  if (e != cudaSuccess) return e;
  const long long heads = (long long)a.batch * a.H;
  const int grid = (int)std::min<long long>(heads, dev.sms);
  kern<<<grid, 32 * (kFGroups * a.GU + 1 + c.NP), c.smem, st>>>(a);
  return cudaGetLastError();
}

template <int DK, typename TS, typename TI, bool KDA>
cudaError_t launch_fused_k(const DFused& a, cudaStream_t st) {
  if (a.K == 1) return launch_fused<DK, TS, TI, KDA, 1>(a, st);
  if (a.K <= 4) return launch_fused<DK, TS, TI, KDA, 4>(a, st);
  return launch_fused<DK, TS, TI, KDA, 8>(a, st);
}

cudaError_t launch_delta(const replayssm_dims& d, const replayssm_state& s, int K, int commit,
                         const void* q, const void* k, const void* v, const float* alpha,
                         const float* beta, float scale, float* o, cudaStream_t st,
                         int32_t* flags = nullptr) {
  DFused a{d.batch, d.heads, d.dv, d.window, K, commit, 0, 0, 0, 0, 0, 0, 0,
           s.S_read ? (const void*)s.S_read : (const void*)s.S_ckpt,
           q, k, v, alpha, beta, scale, o,
           s.ring_q, s.ring_k, s.ring_v, s.ring_alpha, s.ring_beta,
           s.ring_head, s.ring_len, s.status, s.sync, flags};
  const bool rd16 = s.S_read != nullptr, in16 = d.in_dtype == REPLAYSSM_BF16;
  const bool kda = d.kind == REPLAYSSM_KDA;
  // (delta_kernel_config repeats this choice, and launch_fused's, by sizes
  // alone for the host-side query: a change here goes there too)
  if (gram_eligible(d, s, K)) {
    bool launched = false;
    const bf16* S = reinterpret_cast<const bf16*>(s.S_read);
    cudaError_t e;
    if (d.dk == 128)
      e = K == 1 ? launch_gram<128, 1>(a, S, st, launched)
                 : K <= 4 ? launch_gram<128, 4>(a, S, st, launched) : launch_gram<128, 8>(a, S, st, launched);
    else
      e = K == 1 ? launch_gram<64, 1>(a, S, st, launched)
                 : K <= 4 ? launch_gram<64, 4>(a, S, st, launched) : launch_gram<64, 8>(a, S, st, launched);
    if (e != cudaSuccess || launched) return e;
  }
#define RS_FUSED(DK_, TS_)                                                                     \
  return in16 ? (kda ? launch_fused_k<DK_, TS_, bf16, true>(a, st)                             \
                     : launch_fused_k<DK_, TS_, bf16, false>(a, st))                           \
              : (kda ? launch_fused_k<DK_, TS_, float, true>(a, st)                            \
                     : launch_fused_k<DK_, TS_, float, false>(a, st));
  if (d.dk == 128) {
    if (rd16) { RS_FUSED(128, bf16) }
    RS_FUSED(128, float)
  }
  if (rd16) { RS_FUSED(64, bf16) }
  RS_FUSED(64, float)
#undef RS_FUSED
}

}  // namespace

size_t delta_fused_smem(const replayssm_dims& d, int K, bool read16) {
  // the smallest fused block that runs (one prep warp, one stage per group)
  const int ti = d.in_dtype == REPLAYSSM_BF16 ? 2 : 4, ts = read16 ? 2 : 4;
  const int RB = fused_rows(d.dk, ts, d.dv);
  return DFusedSmem(RB, d.dk, d.dv, d.window, K, kFGroups, vector_slots(1, d.dv / RB), 1, 1,
                    d.kind == REPLAYSSM_KDA, ts, ti).total + 1024;
}

bool delta_kernel_config(const replayssm_dims& d, int K, bool read16, size_t optin,
                         replayssm_delta_config& out) {
  // The choice launch_delta makes, by sizes alone: the tensor-core kernel
  // where gram_eligible admits the sizes and gram_config fits, else the
  // fused kernel as launch_fused configures it.
  out = replayssm_delta_config{};
  const bool kda = d.kind == REPLAYSSM_KDA, in16 = d.in_dtype == REPLAYSSM_BF16;
  const char* env = std::getenv("REPLAYSSM_DELTA_TENSOR_CORES");
  const bool tc = !(env && env[0] == '0');
  if (tc && K >= 2 && d.kind == REPLAYSSM_GDN && read16 && in16 && (d.dk == 64 || d.dk == 128) &&
      d.dv % kGRows == 0 && d.window <= kGramN && K <= kGramQ) {
    const GramConfig c = gram_config(d.dk, d.dv, d.window, K, optin);
    if (c.NP > 0) {
      out.tensor_cores = 1;
      out.prep_warps = c.NP;
      out.depth = c.depth;
      out.state_stages = c.NS;
      out.vector_slots = c.NP * c.depth;
      out.consumer_groups = kGGroups;
      out.consumer_warps_per_group = 2;
      out.rows_per_unit = kGRows;
      out.units_per_head = d.dv / kGRows;
      out.threads = 32 * (2 * kGGroups + 1 + c.NP);
      out.smem_bytes = (int64_t)c.smem;
      return true;
    }
  }
  const int ts = read16 ? 2 : 4, ti = in16 ? 2 : 4;
  const int RB = fused_rows(d.dk, ts, d.dv);
  int GU = RB % 64 == 0 ? 2 : 1;
  const int KMAX = K == 1 ? 1 : K <= 4 ? 4 : 8;
  if (RB / GU > 128 || K > KMAX) return false;
  FusedConfig c{0, 0, 0, 0, 0};
  if (K == 1 && ts == 2) c = decode_config(RB, d.dk, d.dv, d.window, kda, ti, optin, GU);
  if (c.NP == 0) c = fused_config(RB, d.dk, d.dv, d.window, K, GU, kda, ts, ti, optin);
  if (c.NP == 0) return false;
  out.prep_warps = c.NP;
  out.depth = c.depth;
  out.state_stages = c.NS;
  out.vector_slots = c.NSL;
  out.consumer_groups = kFGroups;
  out.consumer_warps_per_group = GU;
  out.rows_per_unit = RB;
  out.units_per_head = d.dv / RB;
  out.threads = 32 * (kFGroups * GU + 1 + c.NP);
  out.smem_bytes = (int64_t)c.smem;
  return true;
}

cudaError_t launch_delta_decode(const replayssm_dims& d, const replayssm_state& s, const void* q,
                                const void* k, const void* v, const float* alpha,
                                const float* beta, float scale, float* o, cudaStream_t st) {
  return launch_delta(d, s, 1, 1, q, k, v, alpha, beta, scale, o, st);
}

cudaError_t launch_delta_verify(const replayssm_dims& d, const replayssm_state& s, int K,
                                const void* q, const void* k, const void* v, const float* alpha,
                                const float* beta, float scale, float* o, cudaStream_t st) {
  return launch_delta(d, s, K, 0, q, k, v, alpha, beta, scale, o, st);
}

namespace {

// The consolidate grid; with `step` (its token and flag fields set) the
// fused step's fold + decode of the flagged sequences.
cudaError_t launch_delta_fold_grid(const replayssm_dims& d, const replayssm_state& s, int k_next,
                                   int force, const DFold* step, cudaStream_t st) {
  DFold a{};
  if (step) a = *step;
  a.batch = d.batch;
  a.H = d.heads;
  a.DV = d.dv;
  a.W = d.window;
  a.k_next = k_next;
  a.force = force;
  a.S = s.S_ckpt;
  a.Sr = reinterpret_cast<bf16*>(s.S_read);
  a.ring_k = s.ring_k;
  a.ring_v = s.ring_v;
  a.ring_alpha = s.ring_alpha;
  a.ring_beta = s.ring_beta;
  a.head = s.ring_head;
  a.len = s.ring_len;
  a.status = s.status;
  a.sync = s.sync;
  const bool kda = d.kind == REPLAYSSM_KDA;
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  const DeviceInfo& dev = device_info();
  const long long heads = (long long)d.batch * d.heads;
  const int grid = (int)std::max<long long>((heads + kMaxFoldTiles - 1) / kMaxFoldTiles,
                                            std::min<long long>(heads, (long long)dev.sms * 2));
  // The prefetching form where two of its blocks fit on an SM (static fold
  // list and the per-block reservation included), else the synchronous one.
  const DFoldSmem L(d.dk, d.dv, d.window, in16 ? 2 : 4, kda);
  const bool prefetch = 2 * (L.total + sizeof(FoldList) + 1024) <= (size_t)dev.smem_sm;
  void (*kern)(const DFold);
  size_t smem;
  if (prefetch) {
    smem = L.total;
    if (d.dk == 128)
      kern = in16 ? (kda ? delta_fold_stream_kernel<128, bf16, true> : delta_fold_stream_kernel<128, bf16, false>)
                  : (kda ? delta_fold_stream_kernel<128, float, true> : delta_fold_stream_kernel<128, float, false>);
    else
      kern = in16 ? (kda ? delta_fold_stream_kernel<64, bf16, true> : delta_fold_stream_kernel<64, bf16, false>)
                  : (kda ? delta_fold_stream_kernel<64, float, true> : delta_fold_stream_kernel<64, float, false>);
  } else {
    smem = 4 * (align_up((size_t)d.window * d.dk + align_up((size_t)d.window * (kda ? d.dk : 1), 4) +
                             (size_t)d.window * d.dv + 2 * (size_t)d.window, 4) +
                d.dk + d.dv + 4);
    if (d.dk == 128)
      kern = in16 ? (kda ? delta_fold_kernel<128, bf16, true> : delta_fold_kernel<128, bf16, false>)
                  : (kda ? delta_fold_kernel<128, float, true> : delta_fold_kernel<128, float, false>);
    else
      kern = in16 ? (kda ? delta_fold_kernel<64, bf16, true> : delta_fold_kernel<64, bf16, false>)
                  : (kda ? delta_fold_kernel<64, float, true> : delta_fold_kernel<64, float, false>);
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (!step) {
    kern<<<grid, kDFoldThreads, smem, st>>>(a);
    return cudaGetLastError();
  }
  // the fused step: a programmatic dependent of the decode grid
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDFoldThreads);
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

cudaError_t launch_delta_fold(const replayssm_dims& d, const replayssm_state& s, int k_next,
                              int force, cudaStream_t st) {
  return launch_delta_fold_grid(d, s, k_next, force, nullptr, st);
}

cudaError_t launch_delta_fold_decode(const replayssm_dims& d, const replayssm_state& s,
                                     const void* q, const void* k, const void* v,
                                     const float* alpha, const float* beta, float scale, float* o,
                                     cudaStream_t st) {
  // The decode grid decodes every sequence with room and flags the full
  // rings (state.work holds the flags: the delta kinds use no other
  // workspace); the fold grid then folds exactly those and decodes their
  // token from the new rows.
  int32_t* flags = reinterpret_cast<int32_t*>(s.work);
  cudaError_t e = launch_delta(d, s, 1, 1, q, k, v, alpha, beta, scale, o, st, flags);
  if (e != cudaSuccess) return e;
  DFold step{};
  step.flags = flags;
  step.q = q;
  step.k = k;
  step.v = v;
  step.alpha = alpha;
  step.beta = beta;
  step.scale = scale;
  step.o = o;
  step.ring_q = s.ring_q;
  step.ring_kw = s.ring_k;
  step.ring_vw = s.ring_v;
  step.ring_alphaw = s.ring_alpha;
  step.ring_betaw = s.ring_beta;
  return launch_delta_fold_grid(d, s, 1, 0, &step, st);
}

cudaError_t launch_delta_conventional_verify(const replayssm_dims& d, const float* S, int K,
                                             const void* q, const void* k, const void* v,
                                             const float* alpha, const float* beta, float scale,
                                             float* snap, float* o, cudaStream_t st) {
  DConvSpec a{d.batch, d.heads, d.dv, K, S, q, k, v, alpha, beta, scale, snap, o};
  const long long warps = (long long)d.batch * d.heads * (d.dv / 8);
  const unsigned grid = (unsigned)((warps + kWarps - 1) / kWarps);
  const bool in16 = d.in_dtype == REPLAYSSM_BF16;
  const bool kda = d.kind == REPLAYSSM_KDA;
  void (*kern)(const DConvSpec);
  if (d.dk == 128)
    kern = in16 ? (kda ? delta_conventional_verify_kernel<128, bf16, true> : delta_conventional_verify_kernel<128, bf16, false>)
                : (kda ? delta_conventional_verify_kernel<128, float, true> : delta_conventional_verify_kernel<128, float, false>);
  else
    kern = in16 ? (kda ? delta_conventional_verify_kernel<64, bf16, true> : delta_conventional_verify_kernel<64, bf16, false>)
                : (kda ? delta_conventional_verify_kernel<64, float, true> : delta_conventional_verify_kernel<64, float, false>);
  kern<<<grid, kThreads, 0, st>>>(a);
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
