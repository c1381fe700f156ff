// Tensor-core form of the Gated DeltaNet replay decode and speculative
// verify (BF16 read copy, BF16 inputs, windows of at most kGramN entries).
// Included by delta.cu inside its anonymous namespace.
//
// The backward sweep of query t over the entries 0..top (top = len + t),
//   u <- scale q_t; for i = top..0: c_i = beta_i (k_i . u); u <- alpha_i (u - c_i k_i),
// ends in u_t = A_top scale q_t - sum_i c_{t,i} A_i k_i with A_i = alpha_0 ... alpha_i,
// and the output is o_t = S u_t + sum_i c_{t,i} v_i ("NVIDIA y Princeton aceleran
// modelos híbridos…", paragraphs 2 and 3: replay from the checkpoint, one state
// read for all drafts). So the state is needed only through the products
//   Y = S [q_0 .. q_{K-1} | k_0 .. k_{n-1}]^T        (DV x (K + n)),
// a small dense contraction that the consumers run on the tensor cores as
// soon as a head's entries are staged, independently of the coefficients:
//   o_t = sum_col w_{t,col} Y[:, col] + sum_i c_{t,i} v_i,
//   w_{t,t} = A_top scale,  w_{t,K+i} = -c_{t,i} A_i (i <= top), other weights 0.
// The prep warps get the coefficients c from the Gram form of the sweeps
// (gram_coefficients): a tensor-core tile of key dots and scalar updates.
//
// Roles of the persistent block (one per SM, contiguous heads):
//  - producer warp: streams the state in units of kGRows rows with 2-D
//    tensor-map copies (128-byte swizzle: ldmatrix reads without bank
//    conflicts) into NS stages;
//  - NP prep warps: stage a head's queries, keys, values, gates and betas
//    (cp.async; key and query rows padded to 16 + 2 DK bytes), signal
//    "data", compute the weights, signal "coefficients", append the call's
//    entries to the ring and count the arrivals (decode: the last one
//    commits len + 1);
//  - kGGroups groups of two consumer warps (32 rows each): wait for "data"
//    and the state unit, run the mma.sync m16n8k16 products, release the
//    state stage, wait for "coefficients", combine and write o.
// Every wait is bounded; a timeout sets REPLAYSSM_SEQ_TIMEOUT and ends the
// block after its copies in flight have landed.

constexpr int kGRows = 64;    // state rows per unit
constexpr int kGGroups = 4;   // consumer groups of two warps
constexpr int kGCols = 24;    // columns of Y: K queries then n keys (at most 3 n-tiles)
constexpr int kGMaxWarps = 1 + 2 * kGGroups + 7;

struct alignas(128) DGram {
  CUtensorMap tmap;           // read copy as [batch * H * DV rows, DK] BF16, box [64, kGRows]
  DFused f;                   // call description; RB = kGRows, NS, NP, depth set by the launcher
};

// One prep stage (byte offsets): header (len, head, ok, seq), the vector
// rows [K + W][ks] (queries, then the entries' keys), value rows [W][DV],
// gates [W], betas [W], column weights [K][kGCols], value terms
// e_t = sum_i c_{t,i} v_i [K][DV].
struct GStage {
  size_t ks, vec, vr, ar, br, wc, ev, bytes;
  __host__ __device__ GStage(int DK, int DV, int W, int K) {
    ks = (size_t)DK * 2 + 16;
    vec = 16;
    vr = align_up(vec + (size_t)(K + W) * ks, 16);
    ar = align_up(vr + (size_t)W * DV * 2, 16);
    br = ar + align_up((size_t)W * 4, 16);
    wc = br + align_up((size_t)W * 4, 16);
    ev = wc + (size_t)K * kGCols * 4;
    bytes = align_up(ev + (size_t)K * DV * 4, 128);
  }
};

// Shared memory: NS state stages (1024-byte aligned for the swizzle), their
// barriers, NP x depth prep stages with three barriers each (data,
// coefficients, released), and one Gram scratch per prep warp.
struct GSmem {
  size_t stage, bars, prep, pbars, scratch, total;
  __host__ __device__ GSmem(int DK, int DV, int W, int K, int NS, int NP, int depth) {
    stage = (size_t)kGRows * DK * 2;                      // a multiple of 1024
    bars = (size_t)NS * stage;
    prep = align_up(bars + 16 * (size_t)NS, 128);
    pbars = prep + (size_t)NP * depth * GStage(DK, DV, W, K).bytes;
    scratch = align_up(pbars + 24 * (size_t)NP * depth, 128);
    total = scratch + (size_t)NP * gram_scratch_bytes(K) + 1024;  // + alignment slack
  }
  __host__ __device__ static size_t gram_scratch_bytes(int K) {
    return align_up((size_t)kGramN * kGramT * 4 + (size_t)K * kGramN * 4, 128);
  }
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

template <int DK, int KMAX>
__global__ void __launch_bounds__(32 * kGMaxWarps, 1) delta_gram_kernel(const __grid_constant__ DGram g) {
  extern __shared__ unsigned char smem_raw[];
  const DFused& a = g.f;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int CW = 2 * kGGroups;
  const int NS = a.NS, NP = a.NP, depth = a.depth;
  const int H = a.H, DV = a.DV, K = a.K, W = a.W, nrb = a.nrb;
  // 1024-byte aligned base (the dynamic window follows the static variables)
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const GSmem L(DK, DV, W, K, NS, NP, depth);
  const GStage SG(DK, DV, W, K);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + NS;
  uint64_t* pb = reinterpret_cast<uint64_t*>(smem + L.pbars);  // [NP * depth][3]
  auto pstage = [&](int pw, int d) { return smem + L.prep + ((size_t)pw * depth + d) * SG.bytes; };
  auto dbar = [&](int pw, int d, int k) { return pb + ((size_t)pw * depth + d) * 3 + k; };
  __shared__ int abort_smem;
  volatile int& abort_flag = abort_smem;
  const long long heads = (long long)a.batch * H;
  const int hb0 = (int)(heads * blockIdx.x / gridDim.x);
  const int hb1 = (int)(heads * (blockIdx.x + 1) / gridDim.x);
  const int nh = hb1 - hb0, nu = nh * nrb;
  constexpr uint32_t tile_bytes = (uint32_t)kGRows * DK * 2;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);
    }
    for (int i = 0; i < NP * depth; ++i) {
      mbar_init(pb + 3 * i + 0, 32);        // data staged (every prep lane, after its copies)
      mbar_init(pb + 3 * i + 1, 32);        // coefficients written (every prep lane)
      mbar_init(pb + 3 * i + 2, 2 * nrb);   // released by the head's consumer warps
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  // Refused sequences (pointers out of range, no room for K entries; with
  // a.flags the full rings left to the fold grid): their state rows are not
  // read. Read before any prep warp of the block runs (as in the fused
  // kernel): the last arrival of such a sequence needs this block's heads.
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
    int ps = 0;
    uint32_t pk = 0;
    bool pwrap = false;
    int li = 0, rb = 0;
    bool skip = false;
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
        const int i = (hb0 + li) / H - seq_lo;
        skip = use_skip && ((skipmask[i / 32] >> (i % 32)) & 1u) != 0;
      }
      if (lane == 0) {
        if (skip) {
          mbar_arrive(&full[s]);
        } else {
          mbar_arrive_expect_tx(&full[s], tile_bytes);
          const int row = (hb0 + li) * DV + rb * kGRows;
#pragma unroll
          for (int box = 0; box < DK / 64; ++box)
            tma_load_2d(smem + (size_t)s * L.stage + (size_t)box * kGRows * 128, &g.tmap, box * 64,
                        row, &full[s], pol);
        }
      }
      if (++rb == nrb) {
        rb = 0;
        ++li;
      }
    }
  } else if (warp < CW) {
    // ------------------------------------------------------------ consumers
    const int gi = warp >> 1, part = warp & 1;
    const int gq = lane >> 2, t4 = lane & 3;
    int s = gi;
    uint32_t ph = 0;
    for (int ul = gi; ul < nu; ul += kGGroups) {
      const int li = ul / nrb, rb = ul - li * nrb;
      const int hg = hb0 + li, seq = hg / H, h = hg - seq * H;
      const int pw = li % NP, d = (li / NP) % depth;
      const uint32_t par = (uint32_t)((li / NP) / depth) & 1u;
      const unsigned char* st = pstage(pw, d);
      const bool aborted0 = __shfl_sync(kFull, abort_flag, 0) != 0;
      const bool staged = !aborted0 && mbar_wait_warp(dbar(pw, d, 0), par);
      if (!aborted0 && !staged && lane == 0) {
        abort_flag = 1;
        atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
      }
      if (!staged) break;
      const int* hdr = reinterpret_cast<const int*>(st);
      const int len = hdr[0];
      const bool ok = hdr[2] != 0;
      const int n = len + K, ncols = K + n;
      const bool landed = mbar_wait_warp(&full[s], ph);
      if (!landed) {
        if (lane == 0) {
          abort_flag = 1;
          atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
        }
        break;
      }
      // Y[r][col] for this warp's 32 rows: acc[mt][nt] covers rows
      // 16 mt + gq (+ 8) and columns 8 nt + 2 t4 (+ 1)
      float acc[2][3][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 3; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
      if (ok) {
        const int nts = (ncols + 7) >> 3;
        const uint32_t tile = smem_u32(smem + (size_t)s * L.stage);
        const int mi = lane >> 3;
        // B rows (columns of Y): lane gives row 8 nt + lane % 8 of the vector
        // rows (clamped to a staged row), 16-byte half (lane / 8) % 2, and
        // k-step kk + lane / 16 (x4: two k-steps at once)
        const uint32_t vbase = smem_u32(st + SG.vec) + ((lane >> 3) & 1) * 16 + (lane >> 4) * 32;
#pragma unroll
        for (int kk = 0; kk < DK / 16; kk += 2) {
          uint32_t bfr[3][4];
#pragma unroll
          for (int nt = 0; nt < 3; ++nt) {
            if (nt < nts) {
              const int rowv = min(nt * 8 + (lane & 7), ncols - 1);
              ldsm_x4(bfr[nt], vbase + rowv * (uint32_t)SG.ks + kk * 32);
            }
          }
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int k = kk + k2;
            const int box = k >> 2, c0 = (k & 3) * 2;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              const int r = part * 32 + mt * 16 + (mi & 1) * 8 + (lane & 7);
              const int chunk = c0 + (mi >> 1);
              uint32_t afr[4];
              ldsm_x4(afr, tile + box * (kGRows * 128) + r * 128 + ((chunk ^ (r & 7)) << 4));
#pragma unroll
              for (int nt = 0; nt < 3; ++nt)
                if (nt < nts) mma_bf16_16816(acc[mt][nt], afr, bfr[nt][2 * k2], bfr[nt][2 * k2 + 1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // the state rows are no longer needed
      const bool coef = mbar_wait_warp(dbar(pw, d, 1), par);
      if (!coef) {
        if (lane == 0) {
          abort_flag = 1;
          atomicOr(a.status + seq, REPLAYSSM_SEQ_TIMEOUT);
        }
        break;
      }
      if (ok) {
        const float* wc = reinterpret_cast<const float*>(st + SG.wc);
        const float* ev = reinterpret_cast<const float*>(st + SG.ev);
        const int row0 = rb * kGRows + part * 32;  // first value row of this warp
        float* ybase = a.o + ((size_t)seq * K * H + h) * DV + row0;
#pragma unroll
        for (int t = 0; t < KMAX; ++t) {
          if (t >= K) break;
          // rows of this lane: gq, gq + 8, gq + 16, gq + 24 (of the warp's 32)
          float pr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int nt = 0; nt < 3; ++nt) {
            const float2 w2 = *reinterpret_cast<const float2*>(wc + t * kGCols + nt * 8 + 2 * t4);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              pr[2 * mt] = fmaf(w2.x, acc[mt][nt][0], fmaf(w2.y, acc[mt][nt][1], pr[2 * mt]));
              pr[2 * mt + 1] = fmaf(w2.x, acc[mt][nt][2], fmaf(w2.y, acc[mt][nt][3], pr[2 * mt + 1]));
            }
          }
          // lane t4 of each 4-lane group ends with the row gq + 8 t4
          const float y = reduce_scatter<4>(pr, lane);
          const int row = gq + 8 * t4;
          ybase[(size_t)t * H * DV + row] = y + ev[t * DV + row0 + row];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(dbar(pw, d, 2));
      s += kGGroups;
      if (s >= NS) {
        s -= NS;
        ph ^= 1;
      }
    }
  } else if (warp - CW - 1 < NP) {
    // ------------------------------------------------------------ prep
    constexpr int kKC = DK * 2 / 16;  // 16-byte chunks of a key row
    constexpr int kKR = 32 / kKC;     // rows per pass of the warp
    const int pw = warp - CW - 1;
    const int Wd = ring_wd(W);
    const size_t krow = (size_t)DK * 2, vrow = (size_t)DV * 2;
    const int vcpr = (int)(vrow / 16);
    float* T = reinterpret_cast<float*>(smem + L.scratch + (size_t)pw * GSmem::gram_scratch_bytes(K));
    float* cgr = T + kGramN * kGramT;
    const int nmine = nh > pw ? (nh - pw + NP - 1) / NP : 0;

    // issue side: stage head i_t of this warp into stage i_t % depth once its
    // previous occupant is released by the consumers
    int i_t = 0, i_loaded = -1, i_len = 0, i_hd = 0;
    bool i_ok = false;
    int i_v = hb0 + pw, i_seq = i_v / H, i_h = i_v - (i_v / H) * H;
    bool failed = false;
    auto issue = [&]() {
      const int d = i_t % depth;
      if (i_t >= depth) {
        const uint32_t par = (uint32_t)(i_t / depth - 1) & 1u;
        const bool aborted = __shfl_sync(kFull, abort_flag, 0) != 0;
        if (aborted || !mbar_wait_warp(dbar(pw, d, 2), par)) {
          if (!aborted && lane == 0) {
            abort_flag = 1;
            atomicOr(a.status + i_seq, REPLAYSSM_SEQ_TIMEOUT);
          }
          failed = true;
          return;
        }
      }
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
      unsigned char* st = pstage(pw, d);
      if (lane == 0) {
        int* hdr = reinterpret_cast<int*>(st);
        hdr[0] = i_len;
        hdr[1] = i_hd;
        hdr[2] = i_ok ? 1 : 0;
        hdr[3] = i_seq;
      }
      if (i_ok) {
        const int n = i_len + K, v = i_v;
        const size_t in0 = (size_t)i_seq * K * H + i_h;
        const size_t instep = (size_t)H;
        const int c = (lane % kKC) * 16;
        const unsigned char* rkh = reinterpret_cast<const unsigned char*>(a.ring_k) + (size_t)v * W * krow;
        const unsigned char* ikh = reinterpret_cast<const unsigned char*>(a.k) + in0 * krow;
        const unsigned char* iqh = reinterpret_cast<const unsigned char*>(a.q) + in0 * krow;
        // vector rows: queries 0..K-1, then keys of entries 0..n-1
        for (int j = lane / kKC; j < K + n; j += kKR) {
          const unsigned char* src;
          if (j < K) {
            src = iqh + (size_t)j * instep * krow;
          } else {
            const int e = j - K, slot = i_hd + e < W ? i_hd + e : i_hd + e - W;
            src = e < i_len ? rkh + slot * krow : ikh + (size_t)(e - i_len) * instep * krow;
          }
          cp_async16(st + SG.vec + j * SG.ks + c, src + c);
        }
        const unsigned char* rvh = reinterpret_cast<const unsigned char*>(a.ring_v) + (size_t)v * W * vrow;
        const unsigned char* ivh = reinterpret_cast<const unsigned char*>(a.v) + in0 * vrow;
        for (int idx = lane; idx < n * vcpr; idx += 32) {
          const int j = idx / vcpr, cv = idx - j * vcpr;
          const int slot = i_hd + j < W ? i_hd + j : i_hd + j - W;
          const unsigned char* src = j < i_len ? rvh + slot * vrow : ivh + (size_t)(j - i_len) * instep * vrow;
          cp_async16(st + SG.vr + j * vrow + cv * 16, src + cv * 16);
        }
        if (lane < n) {
          const int j = lane;
          const int slot = i_hd + j < W ? i_hd + j : i_hd + j - W;
          const size_t rs_ = (size_t)v * Wd + slot, is_ = in0 + (size_t)(j - i_len) * instep;
          cp_async4(st + SG.br + 4 * j, j < i_len ? a.ring_beta + rs_ : a.beta + is_);
          cp_async4(st + SG.ar + 4 * j, j < i_len ? a.ring_alpha + rs_ : a.alpha + is_);
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

    int cur_seq = -1, len = 0, hd = 0, seq_count = 0;
    bool ok = false;
    int h = (hb0 + pw) % H;
    while (i_t < depth - 1 && i_t < nmine && !failed) issue();
    for (int t = 0; t < nmine && !failed; ++t) {
      if (i_t < nmine) {
        issue();
        if (failed) break;
        if (depth == 2)
          cp_async_wait_group<1>();  // head t has landed
        else
          cp_async_wait_all();
      } else {
        cp_async_wait_all();
      }
      __syncwarp();
      const int li = pw + t * NP, v = hb0 + li, d = t % depth;
      unsigned char* st = pstage(pw, d);
      const int* hdr = reinterpret_cast<const int*>(st);
      const int seq = hdr[3];
      if (seq != cur_seq) {
        if (a.commit && cur_seq >= 0 && ok && lane == 0)
          arrive_and_finish(a.sync + cur_seq, seq_count, H, [&] { a.len[cur_seq] = len + 1; });
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
      mbar_arrive(dbar(pw, d, 0));  // this lane's copies have landed
      const float* ar = reinterpret_cast<const float*>(st + SG.ar);
      const float* br = reinterpret_cast<const float*>(st + SG.br);
      if (ok) {
        const int n = len + K;
        gram_coefficients<DK, KMAX>(st + SG.vec + K * SG.ks, st + SG.vec, (uint32_t)SG.ks, ar, br, len,
                                    K, a.scale, T, cgr, lane);
        // A_i = alpha_0 ... alpha_i in lane i
        float Ai = 1.f;
        for (int m = 0; m < n && m <= lane; ++m) Ai *= ar[m];
        float* wc = reinterpret_cast<float*>(st + SG.wc);
        for (int t2 = 0; t2 < K; ++t2) {
          const int top = len + t2;
          const float Atop = __shfl_sync(kFull, Ai, top);
          // column lane: a query column (weight A_top scale on its own query)
          // or key column K + i
          const int i = lane - K;
          const float Ak = __shfl_sync(kFull, Ai, max(i, 0));
          float w = 0.f;
          if (lane < K) w = lane == t2 ? Atop * a.scale : 0.f;
          else if (i <= top) w = -cgr[t2 * kGramN + i] * Ak;
          if (lane < kGCols) wc[t2 * kGCols + lane] = w;
        }
        // e_t[r] = sum_{i <= top_t} c_{t,i} v_i[r]: lane rows r = lane + 32 m,
        // the values read once for every query
        const bf16* vr = reinterpret_cast<const bf16*>(st + SG.vr);
        float* ev = reinterpret_cast<float*>(st + SG.ev);
        for (int r = lane; r < DV; r += 32) {
          float e[KMAX];
#pragma unroll
          for (int t2 = 0; t2 < KMAX; ++t2) e[t2] = 0.f;
          for (int i = 0; i < n; ++i) {
            const float vi = to_f(vr[(size_t)i * DV + r]);
#pragma unroll
            for (int t2 = 0; t2 < KMAX; ++t2)
              if (t2 < K && i <= len + t2) e[t2] = fmaf(cgr[t2 * kGramN + i], vi, e[t2]);
          }
#pragma unroll
          for (int t2 = 0; t2 < KMAX; ++t2)
            if (t2 < K) ev[t2 * DV + r] = e[t2];
        }
      }
      __syncwarp();
      mbar_arrive(dbar(pw, d, 1));
      if (ok) {
        // append the call's entries: slot (head + len + i) mod W
        for (int i = 0; i < K; ++i) {
          const int j = len + i;
          const int slot = hd + j < W ? hd + j : hd + j - W;
          const size_t rr = (size_t)v * W + slot;
          block_copy_warp(reinterpret_cast<unsigned char*>(a.ring_k) + rr * krow,
                          st + SG.vec + (K + j) * SG.ks, (int)krow, lane);
          block_copy_warp(reinterpret_cast<unsigned char*>(a.ring_v) + rr * vrow, st + SG.vr + j * vrow,
                          (int)vrow, lane);
          if (a.ring_q)
            block_copy_warp(reinterpret_cast<unsigned char*>(a.ring_q) + rr * krow,
                            st + SG.vec + i * SG.ks, (int)krow, lane);
          if (lane == 0) {
            a.ring_beta[(size_t)v * Wd + slot] = br[j];
            a.ring_alpha[(size_t)v * Wd + slot] = ar[j];
          }
        }
      }
      h += NP;
      while (h >= H) h -= H;
    }
    cp_async_wait_all();
    if (a.commit && cur_seq >= 0 && ok && lane == 0 && !abort_flag)
      arrive_and_finish(a.sync + cur_seq, seq_count, H, [&] { a.len[cur_seq] = len + 1; });
  }
  __syncthreads();
  // No tensor copy may land after the block exits.
  if (tid == 0 && abort_flag) {
    for (int s = 0; s < NS; ++s) {
      mbar_wait(&full[s], 0);
      mbar_wait(&full[s], 1);
    }
  }
}
