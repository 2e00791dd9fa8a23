// sgmv_tc.cuh -- the tensor-core role of the kernel (fused, shrink-only and expand-only):
// adapter groups with many rows.
//
// Operation (Punica Guide: Multi-Tenant LoRA Serving with SGMV, section "The SGMV Mathematical
// Formulation"; section "Hardware-Level Optimizations in SGMV" for the tensor-core tiles of
// long segments): for the rows of one adapter group,
//     v = x . A_k          (rows x h_in) . (h_in x r)
//     y += scale * v . B_k (rows x r) . (r x h_out)
// computed with tcgen05.mma (fp16 / bf16 operands, fp32 accumulation in tensor memory).
//
// Work: a group is cut into m-tiles of 128 rows (the MMA's M, one TMEM lane per row; rows of
// a group come from all of its segments, in segment order, gathered row by row).  The unit of
// work is a cluster of 4 CTAs (fused and shrink-only forms) or a CTA (expand-only).  With fewer
// m-tiles than units, every m-tile gets its own units, which split its 64-column n-tiles;
// otherwise the (m-tile, n-tile) sequence is cut into equal contiguous ranges.  Within a
// cluster the shrink is split over K: member m multiplies a quarter of h_in, and the partial
// v rows are reduced over distributed shared memory (st.async), each member owning 32 rows.
//
// Roles inside the CTA (288 threads; 416 in the long-batch instantiation):
//   warps 0-3  loaders: fill a ring of 24 KB slots -- x and y rows by TMA (one 128-row box
//              when the tile's rows are consecutive tokens, else boxes of 8 consecutive rows),
//              every other row and the weights by 16-byte cp.async (each thread's copies
//              complete the slot's barrier by themselves) -- in the order the MMA consumes
//              them: per m-tile, this CTA's shrink slots {x rows [128 x 64] (K-major, 128-byte
//              swizzle), A rows [64 x r] (MN-major, 128-byte swizzle)}, then per n-tile one
//              expand slot {B rows [r x 64] (MN-major, 128-byte swizzle), y rows [128 x 64]
//              (swizzled for conflict-free row reads)}.
//   warp 8     lane 0 issues the MMAs; the warp owns the TMEM allocation.
//   warps 4-7  epilogue: v (fp32, TMEM) -> cluster reduction -> scale -> split into a 16-bit
//              high part and a 16-bit low part (v' = hi + lo to ~16 mantissa bits) -> TMEM,
//              the A operand of the expand MMAs (D = hi . B + lo . B); then per n-tile
//              y += D, written back in place in the slot and stored by TMA (8-row boxes of
//              consecutive tokens; other rows by 16-byte stores).
//   warps 9-12 (long-batch instantiation) a second epilogue warpgroup: every other n-tile,
//              with its own D buffer.
// TMEM (256 columns): v fp32 [0, 64), hi [64, 96), lo [96, 128), two D buffers [128, 256).
#pragma once

namespace sgmv {

constexpr int kTcRows = 128;    // rows per m-tile (MMA M = TMEM lanes)
constexpr int kTcK = 64;        // h_in per shrink slot: one 128-byte row of 16-bit elements
constexpr int kTcN = 64;        // h_out per expand slot
constexpr int kTcSlot = 24576;  // bytes per ring slot
constexpr int kTcXBytes = kTcRows * 128;  // x part of a shrink slot / y part of an expand slot
constexpr uint32_t kTcCols = 256;
constexpr uint32_t kTmV = 0, kTmHi = 64, kTmLo = 96, kTmD = 128;
constexpr int kTcLoaders = 128;
constexpr int kTcEpi = 128;

// Fixed barriers after the 2 * slots ring barriers.
enum TcBar : int { kTcVFull = 0, kTcVFree, kTcHReady, kTcHFree, kTcDFull0, kTcDFull1,
                   kTcDEmpty0, kTcDEmpty1, kTcRtFull0, kTcRtFull1, kTcRtFree0, kTcRtFree1,
                   kTcRsFull, kTcAgFull, kTcNever, kTcDrain, kTcNumFixed };

// Split-K exchange between the 4 CTAs of a cluster, per round of 16 columns of v:
// reduce-scatter buffer [3 senders][32 rows][16 fp32] and all-gather buffer
// [3 owners][32 rows][16 hi + 16 lo 16-bit values].
constexpr int kTcRowBytes = 64;
constexpr int kTcHalfXchg = 3 * 32 * kTcRowBytes;  // 6144
constexpr int kTcXchgBytes = 2 * kTcHalfXchg;

// Byte offset of 16-byte chunk c of row m inside a block of 128-byte rows in the 128-byte
// swizzle pattern (8-row atoms of 1024 bytes).
static __device__ __forceinline__ uint32_t sw128(int m, int c) {
  return static_cast<uint32_t>((m >> 3) * 1024 + (m & 7) * 128 + ((c ^ (m & 7)) << 4));
}

// One warp: the token index of each of the 128 rows of m-tile [p0, p0 + 128) of the group led
// by segment `lead` (-1 past the group's end).
static __device__ __forceinline__ void tile_rows(const Params& p, const int* starts,
                                                 const int* adapters, int S, int lead, int p0,
                                                 int p_hi, int* out) {
  const int lane = threadIdx.x & 31;
  const int k = adapters[lead];
  if (p.rowmap) {  // a plan's group is one segment: its rows are consecutive in the row map
    for (int q = lane; q < kTcRows; q += 32)
      out[q] = p0 + q < p_hi ? __ldg(p.rowmap + starts[lead] + p0 + q) : -1;
    __syncwarp();
    return;
  }
  for (int q = lane; q < kTcRows; q += 32) out[q] = -1;
  __syncwarp();
  int pos = 0;
  for (int jb = lead; jb < S && pos < p_hi; jb += 32) {
    const int j = jb + lane;
    int len = 0;
    if (j < S && adapters[j] == k) len = max(starts[j + 1] - starts[j], 0);
    int incl = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int seg_lo = pos + incl - len;
    const int a = max(seg_lo, p0), b = min(pos + incl, p_hi);
    for (int q = a; q < b; ++q) out[q - p0] = row_of(p, starts[j] + (q - seg_lo));
    pos += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();
}

// A bounded wait taken by all 32 lanes together: if any lane gives up, every lane does, so
// that no warp-collective instruction (tcgen05.ld / st, shuffles) runs on a partial warp.
static __device__ __forceinline__ bool wwait(const Waiter& w, uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, w.wait<false>(bar, parity));
}

// The same, for barriers that other CTAs of the cluster complete (acquire at cluster scope).
static __device__ __forceinline__ bool wwait_cluster(const Waiter& w, uint32_t bar,
                                                     uint32_t parity) {
  return __all_sync(0xffffffffu, w.wait<true>(bar, parity));
}

// The m-tiles of the CTA's (or, with the split-K shrink, its cluster's) range, walked
// identically by all roles.  With the split, member cr takes quarter cr of each n-tile range.
struct TcWalk {
  int u, u1;       // current / end position in the (m-tile, n-tile) sequence
  int ntile;       // n-tiles per m-tile
  int split, cr;   // split-K cluster member cr of 4, or 0
  int mi, a, b;    // current m-tile and this CTA's n-tile range [a, b) (may be empty)
  __device__ __forceinline__ bool next() {
    if (u >= u1) return false;
    mi = u / ntile;
    const int ca = u - mi * ntile;
    const int cb = min(ntile, ca + (u1 - u));
    u += cb - ca;
    a = split ? ca + (cb - ca) * cr / 4 : ca;
    b = split ? ca + (cb - ca) * (cr + 1) / 4 : cb;
    return true;
  }
};

template <typename T, int R, int MODE, int NT>
struct TcRole {
  // Fused: shrink, v kept in TMEM, expand.  Shrink only: v rows written to v_out (fp32).
  // Expand only: v rows read from v_in (fp32) into TMEM, then the expand.
  static constexpr bool kDoShrink = MODE != kExpand;
  static constexpr bool kDoExpand = MODE != kShrink;
  static_assert(sizeof(T) == 2 && R >= 16 && R <= 64, "tensor role: 16-bit types, r >= 16");
  static constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  // Shrink: N = 64 columns of v (columns >= r are never read).  Expand: N = 64 columns of y.
  static constexpr uint32_t kIdShrink = idesc_f16(kBf16, true, kTcRows, 64);
  static constexpr uint32_t kIdExpand = idesc_f16(kBf16, true, kTcRows, kTcN);
  // Epilogue warpgroups: the wide (long-batch) instantiation has a second one (warps 9-12)
  // that takes every other n-tile and owns the second D buffer; the first one (warps 4-7) also
  // does the per-m-tile work (v exchange, hi / lo into TMEM).
  static constexpr int kGroups = (NT == kThreadsWide && kDoExpand) ? 2 : 1;
  static constexpr int kASlotOff = kTcXBytes;  // A rows follow the x rows in a shrink slot
  static constexpr int kYSlotOff = 8192;       // y rows follow the B rows in an expand slot

  struct Ctx {
    uint32_t bars, ring;
    int slots;
    int* rowtok;  // [2][128]
    uint32_t xchg;   // split-K exchange buffers
    int cr, split;   // cluster member, split-K shrink on
    int k_lo, k_hi;  // this CTA's shrink chunks
    int S;           // segments (or plan groups) in the table
    int* tmask;   // [2]: 8-row blocks moved as one TMA box
    const int *starts, *adapters, *gcnt, *tbase;
    __device__ __forceinline__ uint32_t full(int s) const { return bars + 8u * s; }
    __device__ __forceinline__ uint32_t empty(int s) const { return bars + 8u * (slots + s); }
    __device__ __forceinline__ uint32_t fx(int b) const { return bars + 8u * (2 * slots + b); }
    __device__ __forceinline__ uint32_t slot(int s) const {
      return ring + static_cast<uint32_t>(s) * kTcSlot;
    }
    // m-tile -> (lead segment, first group row, rows in the tile)
    __device__ __forceinline__ void tile(int S, int mi, int& lead, int& p0, int& nrow) const {
      int lo = 0, hi = S - 1;  // largest i with tbase[i] <= mi
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tbase[mid] <= mi) lo = mid; else hi = mid - 1;
      }
      lead = lo;
      p0 = (mi - tbase[lo]) * kTcRows;
      nrow = min(kTcRows, gcnt[lo] - p0);
    }
  };

  struct Ring {
    int s;
    uint32_t par;
    __device__ __forceinline__ void next(int slots) {
      if (++s == slots) {
        s = 0;
        par ^= 1u;
      }
    }
  };

  // ------------------------------------------------------------------------ loaders ----
  // Ring slot s is always filled by loader warp s % 4 alone, so that up to four slots are
  // being issued at once (one slot's issue is a chain of dependent barrier, TMA and cp.async
  // instructions; spreading every slot over all four warps left that chain serial).  Binding
  // the warp to the ring slot, not to the sequence number, keeps every use of a slot issued in
  // order by one warp: a parity wait on the slot's "empty" barrier can then never be satisfied
  // by a phase two uses old.
  // Returns, for the drain of a CTA that gives up, the ring slots this warp filled (low 16
  // bits) and the phase parity of each one's last fill (high 16 bits).
  __device__ __forceinline__ static uint32_t loader(const Params& p, const Ctx& c,
                                                    const Waiter& w, TcWalk wk) {
    uint32_t issued = 0, parity = 0;
    const int lt = threadIdx.x;  // 0..127
    const int warp = lt >> 5, lane = lt & 31;
    const T* x = static_cast<const T*>(p.x);
    const T* y = static_cast<const T*>(p.y);
    // x and y may be written by the previous kernel of the stream; the segment table, the row
    // map, the pointer arrays and the weights may not (the launch contract of a programmatic
    // dependent).  So the first m-tile's row table and the weight part of each warp's first
    // slot (never used before: no wait on a consumer) are issued at once, and the activation
    // parts of those slots right after the wait on the previous kernel, which comes before the
    // warp's next slot or at the end of the first m-tile.  One slot per warp: a second one's
    // weight copies would hold back the first one's x copy whenever the previous kernel has
    // already completed (measured on GB300, 8-slot ring: 0.5-0.9 us per call slower; 4-slot
    // ring, 256 rows of one adapter on the tensor cores: 16.7 -> 11.6 us per chained call).
    constexpr int kDefer = 4;  // loader warps
    bool prior_done = !p.dependent;
    uint32_t deferred = 0;  // first-round slots of this warp whose activation part is pending
    int seq = 0;            // position in the slot sequence (every warp counts every slot)
    Ring rg{0, 0};
    bool ok = true;
    for (int li = 0; ok && wk.next(); ++li) {
      const int par = li & 1;
      int lead, p0, nrow;
      c.tile(c.S, wk.mi, lead, p0, nrow);
      int* rt = c.rowtok + par * kTcRows;
      if (warp == 0) {
        if (!wwait(w, c.fx(kTcRtFree0 + par), ((li >> 1) & 1) ^ 1)) break;
        tile_rows(p, c.starts, c.adapters, c.S, lead, p0, p0 + nrow, rt);
        // Rows of consecutive tokens move by TMA: the whole tile as one 128-row box when all
        // 128 rows are consecutive, else each 8-row block of consecutive tokens as one box
        // (one 1024-byte swizzle atom); every other row by cp.async.
        bool run = false, line = false;
        if (lane < kTcRows / 8) {
          const int t0 = rt[8 * lane];
          run = t0 >= 0;
#pragma unroll
          for (int j = 1; j < 8; ++j) run = run && rt[8 * lane + j] == t0 + j;
          line = run && t0 == rt[0] + 8 * lane;
        }
        uint32_t mask = __ballot_sync(0xffffffffu, run);
        if (__ballot_sync(0xffffffffu, line) == 0xffffu) mask |= 1u << 16;
        // A shorter tile whose nrow rows are one run of consecutive tokens (a segment's end):
        // its full 8-row blocks move by at most four boxes of 64 / 32 / 16 / 8 rows.
        bool pre = true;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int m = lane + 32 * i;
          pre = pre && (m >= nrow || rt[m] == rt[0] + m);
        }
        if (!((mask >> 16) & 1u) && nrow >= 8 && __all_sync(0xffffffffu, pre))
          mask |= 1u << 17;
        if (lane == 0) {
          c.tmask[par] = static_cast<int>(mask);
          mbar_arrive(c.fx(kTcRtFull0 + par));
        }
      }
      // Every loader warp takes every table hand-off in order and releases the table when it
      // is done with it (the table's "free" barrier counts the four loader warps too), so that
      // no warp can run ahead of, or fall two phases behind, the table barriers -- even a warp
      // that fills no slot of this m-tile.
      if (!wwait(w, c.fx(kTcRtFull0 + par), (li >> 1) & 1)) break;
      const int nsh = c.k_hi - c.k_lo;  // shrink slots of the m-tile (they come first)
      const int n_sl = nsh + (kDoExpand ? wk.b - wk.a : 0);
      bool mine = false;
      for (int i = 0, sl = rg.s; i < min(n_sl, c.slots); ++i) {
        mine = mine || (sl & 3) == warp;
        if (++sl == c.slots) sl = 0;
      }
      if (!mine) {
        for (int i = 0; i < n_sl; ++i) rg.next(c.slots);
        seq += n_sl;
        __syncwarp();
        if (lane == 0) mbar_arrive(c.fx(kTcRtFree0 + par));
        continue;
      }
      const uint32_t mask = static_cast<uint32_t>(c.tmask[par]);
      const bool whole = (mask >> 16) & 1u;
      const bool all_boxes = whole || (mask & 0xffffu) == 0xffffu;
      const uint32_t tx = whole ? 128u * 128u : static_cast<uint32_t>(__popc(mask & 0xffffu)) * 1024u;
      const bool run_tile = (mask >> 17) & 1u;
      // 8-row box `lane` (gathered tiles), or for a run tile the box of 64 >> (lane - 1) rows
      // (lanes 1-4, when that bit of the run's full-block length is set; larger boxes first)
      int pbox = 0, prow = 0;
      if (run_tile && lane >= 1 && lane <= 4) {
        const int nb = nrow & ~7;
        const int sz = 128 >> lane;
        if (nb & sz) {
          pbox = sz;
          prow = nb & ~(2 * sz - 1);
        }
      }
      const bool my_box = !whole && !run_tile && lane < 16 && ((mask >> lane) & 1u);
      const int box_tok = my_box ? rt[8 * lane] : (pbox ? rt[prow] : 0);
      const int tile_tok = rt[0];
      const int k = c.adapters[lead];
      const int rk = rank_of<R>(p, k);  // A / B hold rk columns / rows; the rest reads as zero
      const T* Ak = kDoShrink ? static_cast<const T*>(p.A_ptrs[k]) +
                                    static_cast<size_t>(p.layer) * p.h_in * rk
                              : nullptr;
      const T* Bk = kDoExpand ? static_cast<const T*>(p.B_ptrs[k]) +
                                    static_cast<size_t>(p.layer) * rk * p.h_out
                              : nullptr;
      // Activation part of a shrink slot (the x rows [128 x 64] of h_in chunk k0) and of an
      // expand slot (the y rows [128 x 64] of h_out chunk n0): the slot's TMA bytes, and each
      // lane's arrival, which covers every cp.async the lane issued before it (weights too).
      auto acts_x = [&](uint32_t dst, uint32_t bar, int k0) {
        if (lane == 0) {
          mbar_arrive_expect_tx(bar, tx);
          if (whole) tma_load_2d(dst, &p.tmap_x128, k0, tile_tok, bar);
        }
        if (my_box) tma_load_2d(dst + 1024u * lane, &p.tmap_x8, k0, box_tok, bar);
        if (pbox) {
          const uint32_t d = dst + 128u * prow;
          if (pbox == 64) tma_load_2d(d, &p.tmap_x64, k0, box_tok, bar);
          else if (pbox == 32) tma_load_2d(d, &p.tmap_x32, k0, box_tok, bar);
          else if (pbox == 16) tma_load_2d(d, &p.tmap_x16, k0, box_tok, bar);
          else tma_load_2d(d, &p.tmap_x8, k0, box_tok, bar);
        }
        if (!all_boxes) {  // rows outside boxes, 16 bytes at a time
          for (int u = lane; u < kTcRows * 8; u += 32) {
            const int m = u >> 3, ch = u & 7;
            const int tok = rt[m];
            if (tok < 0 || ((mask >> (m >> 3)) & 1u)) continue;
            const uint32_t d = dst + sw128(m, ch);
            if (k0 + ch * 8 < p.h_in)
              cp_async16(d, x + static_cast<size_t>(tok) * p.ldx + k0 + ch * 8);
            else
              cp_async16_zero(d, x);
          }
        }
        cp_async_arrive(bar);
      };
      auto acts_y = [&](uint32_t dst, uint32_t bar, int n0) {
        const int nvalid = min(kTcN, p.h_out - n0) >> 3;  // 16-byte chunks in range
        if (lane == 0) {
          mbar_arrive_expect_tx(bar, tx);
          if (whole) tma_load_2d(dst + kYSlotOff, &p.tmap_y128, n0, tile_tok, bar);
        }
        if (my_box) tma_load_2d(dst + kYSlotOff + 1024u * lane, &p.tmap_y8, n0, box_tok, bar);
        if (pbox) {
          const uint32_t d = dst + kYSlotOff + 128u * prow;
          if (pbox == 64) tma_load_2d(d, &p.tmap_y64, n0, box_tok, bar);
          else if (pbox == 32) tma_load_2d(d, &p.tmap_y32, n0, box_tok, bar);
          else if (pbox == 16) tma_load_2d(d, &p.tmap_y16, n0, box_tok, bar);
          else tma_load_2d(d, &p.tmap_y8, n0, box_tok, bar);
        }
        if (!all_boxes) {
          for (int u = lane; u < kTcRows * 8; u += 32) {
            const int m = u >> 3, ch = u & 7;
            const int tok = rt[m];
            if (tok < 0 || ch >= nvalid || ((mask >> (m >> 3)) & 1u)) continue;
            cp_async16(dst + kYSlotOff + sw128(m, ch),
                       y + static_cast<size_t>(tok) * p.ldy + n0 + ch * 8);
          }
        }
        cp_async_arrive(bar);
      };
      // The wait on the previous kernel, then the pending activation parts.  Deferred slots
      // belong to the first round of the first m-tile, where slot s holds sequence position s.
      auto release = [&]() {
        pdl_wait_prior();
        prior_done = true;
        for (int s = 0; s < c.slots; ++s) {
          if (!((deferred >> s) & 1u)) continue;
          if (s < nsh) acts_x(c.slot(s), c.full(s), (c.k_lo + s) * kTcK);
          else acts_y(c.slot(s), c.full(s), (wk.a + s - nsh) * kTcN);
          issued |= 1u << s;
          parity &= ~(1u << s);
        }
        deferred = 0;
      };
      // shrink slots: x rows [128 x 64] + A rows [64 x r]
      for (int kc = c.k_lo; kc < c.k_hi; ++kc, rg.next(c.slots), ++seq) {
        if ((rg.s & 3) != warp) continue;
        const bool defer = !prior_done && li == 0 && seq < min(kDefer, c.slots);
        if (!prior_done && !defer) release();
        if (!wwait(w, c.empty(rg.s), rg.par ^ 1u)) { ok = false; break; }
        const uint32_t dst = c.slot(rg.s), bar = c.full(rg.s);
        const int k0 = kc * kTcK;
        constexpr int kCpr = R / 8;  // 16-byte chunks per A row
        if (rk == R) {  // every unranked call: constant strides
#pragma unroll 4
          for (int u = lane; u < kTcK * kCpr; u += 32) {
            const int kr = u / kCpr, cc = u - kr * kCpr;
            const uint32_t d = dst + kASlotOff + sw128(kr, cc);
            if (k0 + kr < p.h_in)
              cp_async16(d, Ak + static_cast<size_t>(k0 + kr) * R + cc * 8);
            else
              cp_async16_zero(d, Ak);
          }
        } else {
#pragma unroll 4
          for (int u = lane; u < kTcK * kCpr; u += 32) {
            const int kr = u / kCpr, cc = u - kr * kCpr;
            const uint32_t d = dst + kASlotOff + sw128(kr, cc);
            if (k0 + kr < p.h_in && cc * 8 < rk)
              cp_async16(d, Ak + static_cast<size_t>(k0 + kr) * rk + cc * 8);
            else
              cp_async16_zero(d, Ak);
          }
        }
        if (defer) {
          deferred |= 1u << rg.s;
          continue;
        }
        acts_x(dst, bar, k0);
        issued |= 1u << rg.s;
        parity = (parity & ~(1u << rg.s)) | (rg.par << rg.s);
      }
      if (!ok) break;
      // expand slots: B rows [r x 64] + y rows [128 x 64]
      for (int nt = wk.a; kDoExpand && nt < wk.b; ++nt, rg.next(c.slots), ++seq) {
        if ((rg.s & 3) != warp) continue;
        const bool defer = !prior_done && li == 0 && seq < min(kDefer, c.slots);
        if (!prior_done && !defer) release();
        if (!wwait(w, c.empty(rg.s), rg.par ^ 1u)) { ok = false; break; }
        const uint32_t dst = c.slot(rg.s), bar = c.full(rg.s);
        const int n0 = nt * kTcN;
        const int nvalid = min(kTcN, p.h_out - n0) >> 3;  // 16-byte chunks in range
        if (rk == R) {  // every unranked call
#pragma unroll 4
          for (int u = lane; u < R * 8; u += 32) {
            const int kr = u >> 3, cc = u & 7;
            if (cc < nvalid)
              cp_async16(dst + sw128(kr, cc),
                         Bk + static_cast<size_t>(kr) * p.h_out + n0 + cc * 8);
          }
        } else {
#pragma unroll 4
          for (int u = lane; u < R * 8; u += 32) {
            const int kr = u >> 3, cc = u & 7;
            if (kr >= rk)  // past the adapter's rank: zeros (0 x stale data could be NaN)
              cp_async16_zero(dst + sw128(kr, cc), Bk);
            else if (cc < nvalid)
              cp_async16(dst + sw128(kr, cc),
                         Bk + static_cast<size_t>(kr) * p.h_out + n0 + cc * 8);
          }
        }
        if (defer) {
          deferred |= 1u << rg.s;
          continue;
        }
        acts_y(dst, bar, n0);
        issued |= 1u << rg.s;
        parity = (parity & ~(1u << rg.s)) | (rg.par << rg.s);
      }
      // the activation parts still pending (the m-tile ended within the first round): issued
      // before the table is released, since they read it
      if (ok && deferred) release();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.fx(kTcRtFree0 + par));
    }
    cp_async_wait_all();  // every copy lands before the CTA moves on
    return issued | (parity << 16);
  }

  // ---------------------------------------------------------------------- MMA issuer ----
  __device__ __forceinline__ static void issuer(const Params& p, const Ctx& c, const Waiter& w,
                                                TcWalk wk, uint32_t tm) {
    Ring rg{0, 0};
    int dq = 0;
    uint32_t dpar = 0;
    for (int li = 0; wk.next(); ++li) {
      // The previous tile's v has been read out of TMEM -- waited for every tile, even by a
      // split-K member with no chunks to multiply, so that the issuer never runs two phases
      // ahead of the epilogue on the v barriers.
      if (kDoShrink && !w.wait<false>(c.fx(kTcVFree), (li & 1) ^ 1)) return;
      for (int kc = c.k_lo; kc < c.k_hi; ++kc) {
        if (!w.wait<false>(c.full(rg.s), rg.par)) return;
        fence_proxy_async();  // cp.async (generic proxy) data -> the MMA's async-proxy reads
        tc_fence_after();
        const uint32_t sa = c.slot(rg.s);
#pragma unroll
        for (int j = 0; j < kTcK / 16; ++j)
          umma_ss(tm + kTmV, sdesc_sw128(sa + 32u * j, 16, 1024),
                  sdesc_sw128(sa + kASlotOff + 2048u * j, 8192, 1024), kIdShrink,
                  kc != c.k_lo || j != 0);
        umma_commit(c.empty(rg.s));
        mbar_arrive_n(c.empty(rg.s), 4);  // a shrink slot holds no y rows for the epilogue
        rg.next(c.slots);
      }
      if constexpr (kDoShrink) umma_commit(c.fx(kTcVFull));
      if constexpr (!kDoExpand) continue;
      if (!w.wait<false>(c.fx(kTcHReady), li & 1)) return;
      tc_fence_after();
      for (int nt = wk.a; nt < wk.b; ++nt) {
        if (!w.wait<false>(c.full(rg.s), rg.par)) return;
        if (!w.wait<false>(c.fx(kTcDEmpty0 + dq), dpar ^ 1u)) return;
        fence_proxy_async();
        tc_fence_after();
        const uint32_t d = tm + kTmD + 64u * dq;
        const uint32_t sb = c.slot(rg.s);
#pragma unroll
        for (int j = 0; j < R / 16; ++j) {
          const uint64_t bd = sdesc_sw128(sb + 2048u * j, 8192, 1024);
          umma_ts(d, tm + kTmHi + 8u * j, bd, kIdExpand, j != 0);
          umma_ts(d, tm + kTmLo + 8u * j, bd, kIdExpand, 1);
        }
        umma_commit(c.empty(rg.s));
        umma_commit(c.fx(kTcDFull0 + dq));
        rg.next(c.slots);
        if (++dq == 2) {
          dq = 0;
          dpar ^= 1u;
        }
      }
      umma_commit(c.fx(kTcHFree));
    }
  }

  // 16 columns [c0, c0 + 16) of this thread's v row (fp32): shrink only -> v_out; otherwise
  // scale -> 16-bit hi + lo -> TMEM.
  __device__ __forceinline__ static void finish16(const Params& p, uint32_t tq, int c0,
                                                  const uint32_t (&v)[16], int tok_row,
                                                  float sc) {
    if constexpr (MODE == kShrink) {
      if (tok_row >= 0) {
        float4* dst = reinterpret_cast<float4*>(p.v_out + static_cast<size_t>(tok_row) * R + c0);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                               __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
      }
    } else {
      uint32_t hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        split2(sc * __uint_as_float(v[2 * e]), sc * __uint_as_float(v[2 * e + 1]),
               hi[e], lo[e]);
      tmem_st8(tq + kTmHi + c0 / 2, hi);
      tmem_st8(tq + kTmLo + c0 / 2, lo);
    }
  }

  // Split-K shrink: this CTA (member cr of the cluster) holds the partial v of its quarter of
  // h_in for all 128 rows; member q owns rows [32q, 32q + 32).  Per round of 16 columns: every
  // epilogue warp q != cr pushes its rows' partial to member q (st.async, counted on q's
  // reduce barrier); warp cr (the owner) sums the four partials in member order, finishes its
  // rows, and pushes their hi / lo to the other members (counted on their gather barrier; in
  // a shrink, a 4-byte acknowledgement instead).  A warp starts round j + 1 only after the
  // gather barrier of round j completed, which proves that every buffer it writes next has
  // been read.
  __device__ __forceinline__ static bool exchange(const Params& p, const Ctx& c, const Waiter& w,
                                                  uint32_t tq, int q, int lane, int tok_row,
                                                  uint32_t rnd, int* ctl, float sc) {
    const bool has_k = c.k_hi > c.k_lo;
    const uint32_t rs = c.xchg, ag = c.xchg + kTcHalfXchg;
    for (int j = 0; j < R / 16; ++j) {
      const uint32_t ph = (rnd + j) & 1u;
      uint32_t pv[16];
      if (has_k) {
        tmem_ld16(tq + kTmV + 16 * j, pv);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) pv[e] = 0u;
      }
      if (q != c.cr) {
        const int sslot = c.cr < q ? c.cr : c.cr - 1;
        const uint32_t dst = cluster_map(rs + static_cast<uint32_t>((sslot * 32 + lane) * kTcRowBytes), q);
        const uint32_t rb = cluster_map(c.fx(kTcRsFull), q);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          st_async_v4(dst + 16u * e, pv[4 * e], pv[4 * e + 1], pv[4 * e + 2], pv[4 * e + 3], rb);
        if (!wwait_cluster(w, c.fx(kTcAgFull), ph)) return false;
        if constexpr (MODE == kFused) {
          const int tslot = q < c.cr ? q : q - 1;
          const uint32_t src = ag + static_cast<uint32_t>((tslot * 32 + lane) * kTcRowBytes);
          const uint4 h0 = lds128(src), h1 = lds128(src + 16), l0 = lds128(src + 32),
                      l1 = lds128(src + 48);
          const uint32_t hi[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
          const uint32_t lo[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
          tmem_st8(tq + kTmHi + 8 * j, hi);
          tmem_st8(tq + kTmLo + 8 * j, lo);
        }
      } else {
        if (lane == 0) {
          mbar_arrive_expect_tx(c.fx(kTcRsFull), kTcHalfXchg);
          mbar_arrive_expect_tx(c.fx(kTcAgFull), MODE == kFused ? kTcHalfXchg : 3 * 4);
          ctl[kCtlPending] = 1 + static_cast<int>(ph);  // both armed: drained if we give up
        }
        if (!wwait_cluster(w, c.fx(kTcRsFull), ph)) return false;
        float sum[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) sum[e] = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          if (m == c.cr) {
#pragma unroll
            for (int e = 0; e < 16; ++e) sum[e] += __uint_as_float(pv[e]);
          } else {
            const int sl = m < c.cr ? m : m - 1;
            const uint32_t src = rs + static_cast<uint32_t>((sl * 32 + lane) * kTcRowBytes);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint4 t = lds128(src + 16u * e);
              sum[4 * e] += __uint_as_float(t.x);
              sum[4 * e + 1] += __uint_as_float(t.y);
              sum[4 * e + 2] += __uint_as_float(t.z);
              sum[4 * e + 3] += __uint_as_float(t.w);
            }
          }
        }
        uint32_t v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(sum[e]);
        finish16(p, tq, 16 * j, v, tok_row, sc);
        if constexpr (MODE == kFused) {
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            split2(sc * sum[2 * e], sc * sum[2 * e + 1], hi[e], lo[e]);
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            if (pp == c.cr) continue;
            const int tslot = c.cr < pp ? c.cr : c.cr - 1;
            const uint32_t dst =
                cluster_map(ag + static_cast<uint32_t>((tslot * 32 + lane) * kTcRowBytes), pp);
            const uint32_t gb = cluster_map(c.fx(kTcAgFull), pp);
            st_async_v4(dst, hi[0], hi[1], hi[2], hi[3], gb);
            st_async_v4(dst + 16, hi[4], hi[5], hi[6], hi[7], gb);
            st_async_v4(dst + 32, lo[0], lo[1], lo[2], lo[3], gb);
            st_async_v4(dst + 48, lo[4], lo[5], lo[6], lo[7], gb);
          }
        } else if (lane == 0) {
          for (int pp = 0; pp < 4; ++pp)
            if (pp != c.cr)
              st_async_f32(cluster_map(ag, pp), 0.f, cluster_map(c.fx(kTcAgFull), pp));
        }
        if (!wwait_cluster(w, c.fx(kTcAgFull), ph)) return false;
        if (lane == 0) ctl[kCtlPending] = 0;
      }
    }
    return true;
  }

  // ------------------------------------------------------------------------ epilogue ----
  // On every exit, normal or after a wait ran out, this thread's TMA stores have finished
  // reading shared memory before it returns.
  __device__ __forceinline__ static void epilogue(const Params& p, const Ctx& c, const Waiter& w,
                                                  TcWalk wk, uint32_t tm, int g, int* ctl) {
    epilogue_tiles(p, c, w, wk, tm, g, ctl);
    bulk_wait_read();
  }

  __device__ __forceinline__ static void epilogue_tiles(const Params& p, const Ctx& c,
                                                        const Waiter& w, TcWalk wk, uint32_t tm,
                                                        int g, int* ctl) {
    const int q = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;  // TMEM lane quarter, lane
    const int row = q * 32 + lane;                                   // tile row = TMEM lane
    const uint32_t tq = tm + (static_cast<uint32_t>(q * 32) << 16);
    T* y = static_cast<T*>(p.y);
    pdl_wait_prior();
    Ring rg{0, 0};
    // D buffer of the n-tiles this warpgroup takes: the issuer alternates the two buffers over
    // the CTA's n-tile sequence; with two groups, group g owns buffer g (every other n-tile).
    int dq = kGroups == 2 ? g : 0;
    uint32_t dpar = 0;
    uint32_t jn = 0;   // n-tiles of the CTA so far (all groups)
    uint32_t rnd = 0;  // split-K exchange rounds so far (barrier parity)
    for (int li = 0; wk.next(); ++li) {
      const int par = li & 1;
      if (!wwait(w, c.fx(kTcRtFull0 + par), (li >> 1) & 1)) return;
      const int* rt = c.rowtok + par * kTcRows;
      const int tok_row = rt[row];
      volatile int* tile_go = ctl + kCtlTileGo;
      if (kGroups == 2 && g == 1) {
        // The second group skips the per-m-tile work below and would reach this m-tile's first
        // expand slot while the ring is still cycling through its shrink fills: a parity wait
        // on that slot could then see a shrink phase complete and pass two phases early.  It
        // waits first until group 0 has seen every shrink MMA of the m-tile complete (a
        // monotonic counter: no phase aliasing), after which the slot's next completed phase
        // is its expand fill.
        if (!__all_sync(0xffffffffu, w.until(tile_go, li))) return;
      }
      float sc = p.scale;  // the scale of this m-tile's adapter
      if (p.adapter_scale) {
        int lead, p0, nrow;
        c.tile(c.S, wk.mi, lead, p0, nrow);
        sc = scale_of(p, c.adapters[lead]);
      }
      if (g == 0) {  // the per-m-tile work: v into TMEM as hi / lo
        if constexpr (kDoShrink) {
          if (!wwait(w, c.fx(kTcVFull), li & 1)) return;
        }
        if constexpr (kDoExpand) {
          if (!wwait(w, c.fx(kTcHFree), (li & 1) ^ 1)) return;
        }
        if (kGroups == 2 && q == 0 && lane == 0) *tile_go = li;  // shrink slots all consumed
        tc_fence_after();
        if constexpr (kDoShrink) {
          if (c.split) {
            if (!exchange(p, c, w, tq, q, lane, tok_row, rnd, ctl, sc)) return;
            rnd += R / 16;
          } else {
#pragma unroll
            for (int c0 = 0; c0 < R; c0 += 16) {
              uint32_t v[16];
              tmem_ld16(tq + kTmV + c0, v);
              tmem_wait_ld();
              finish16(p, tq, c0, v, tok_row, sc);
            }
          }
        } else {  // expand only: v rows from v_in
#pragma unroll
          for (int c0 = 0; c0 < R; c0 += 16) {
            uint32_t v[16];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
              if (tok_row >= 0)
                f = reinterpret_cast<const float4*>(p.v_in + static_cast<size_t>(tok_row) * R +
                                                    c0)[e];
              v[4 * e] = __float_as_uint(f.x);
              v[4 * e + 1] = __float_as_uint(f.y);
              v[4 * e + 2] = __float_as_uint(f.z);
              v[4 * e + 3] = __float_as_uint(f.w);
            }
            finish16(p, tq, c0, v, tok_row, sc);
          }
        }
        if constexpr (kDoExpand) tmem_wait_st();
        tc_fence_before();
        if constexpr (kDoShrink) mbar_arrive(c.fx(kTcVFree));
        if constexpr (MODE == kShrink) {
          mbar_arrive(c.fx(kTcRtFree0 + par));
          continue;
        }
        mbar_arrive(c.fx(kTcHReady));
      }
      // skip the shrink slots of this m-tile
      for (int kc = c.k_lo; kc < c.k_hi; ++kc) rg.next(c.slots);
      const uint32_t mask = static_cast<uint32_t>(c.tmask[par]);
      int pend = -1;  // ring slot whose TMA stores may still be reading it
      for (int nt = wk.a; nt < wk.b; ++nt, ++jn) {
        if (kGroups == 2 && static_cast<int>(jn & 1u) != g) {  // the other group's n-tile
          rg.next(c.slots);
          continue;
        }
        // y rows of the slot (landed with the slot) into registers while the MMAs run
        if (!wwait(w, c.full(rg.s), rg.par)) return;
        const uint32_t ys = c.slot(rg.s) + kYSlotOff;
        uint4 yv[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) yv[cc] = lds128(ys + sw128(row, cc));
        if (!wwait(w, c.fx(kTcDFull0 + dq), dpar)) return;
        tc_fence_after();
        const int n0 = nt * kTcN;
        const int nvalid = min(kTcN, p.h_out - n0) >> 3;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) yv[cc] = lds128(ys + sw128(row, 4 + cc));
          }
          uint32_t d[32];
          tmem_ld32(tq + kTmD + 64u * dq + 32u * h, d);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            sts128(ys + sw128(row, 4 * h + cc), add8(yv[cc], d + 8 * cc));
        }
        tc_fence_before();
        fence_proxy_async();  // the rows just written are read by TMA stores
        __syncwarp();
        if (lane == 0) mbar_arrive(c.fx(kTcDEmpty0 + dq));
        // this warp's 32 rows = 8-row blocks 4q..4q+3: a block of consecutive tokens leaves by
        // one TMA store (columns past h_out are not written), other rows by 16-byte stores
        const int blk = 4 * q + lane;
        const bool boxed = lane < 4 && ((mask >> blk) & 1u);
        if (boxed) {
          tma_store_2d(&p.tmap_y8, n0, rt[8 * blk], ys + 1024u * blk);
          bulk_commit();
        }
        if ((mask & (0xfu << (4 * q))) != (0xfu << (4 * q))) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = q * 32 + i * 4 + (lane >> 3), cc = lane & 7;
            const int tok = rt[rr];
            if (tok >= 0 && cc < nvalid && !((mask >> (rr >> 3)) & 1u))
              *reinterpret_cast<uint4*>(y + static_cast<size_t>(tok) * p.ldy + n0 + cc * 8) =
                  lds128(ys + sw128(rr, cc));
          }
        }
        // A slot is reused only after its TMA stores have read it: release the previous
        // n-tile's slot now (its stores have had a whole n-tile to read), this one next time.
        if (boxed) bulk_wait_read_1();
        __syncwarp();
        if (lane == 0 && pend >= 0) mbar_arrive(c.empty(pend));
        pend = rg.s;
        rg.next(c.slots);
        if (kGroups == 2) {
          dpar ^= 1u;
        } else if (++dq == 2) {
          dq = 0;
          dpar ^= 1u;
        }
      }
      if (pend >= 0) {  // the m-tile's last slot
        bulk_wait_read();
        __syncwarp();
        if (lane == 0) mbar_arrive(c.empty(pend));
        pend = -1;
      }
      mbar_arrive(c.fx(kTcRtFree0 + par));
    }
  }

  // v' = hi + lo with hi = round(v'), lo = round(v' - hi): two values packed per 32 bits.
  __device__ __forceinline__ static void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    if constexpr (kBf16) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
      const float2 hf = __bfloat1622float2(h);
      const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
      hi = *reinterpret_cast<const uint32_t*>(&h);
      lo = *reinterpret_cast<const uint32_t*>(&l);
    } else {
      const __half2 h = __floats2half2_rn(a, b);
      const float2 hf = __half22float2(h);
      const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
      hi = *reinterpret_cast<const uint32_t*>(&h);
      lo = *reinterpret_cast<const uint32_t*>(&l);
    }
  }

  // Eight 16-bit y values + eight fp32 D values, rounded once.
  __device__ __forceinline__ static uint4 add8(uint4 yv, const uint32_t* d) {
    const uint32_t in[4] = {yv.x, yv.y, yv.z, yv.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (kBf16) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&in[i]));
        const __nv_bfloat162 r = __floats2bfloat162_rn(f.x + __uint_as_float(d[2 * i]),
                                                       f.y + __uint_as_float(d[2 * i + 1]));
        out[i] = *reinterpret_cast<const uint32_t*>(&r);
      } else {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&in[i]));
        const __half2 r = __floats2half2_rn(f.x + __uint_as_float(d[2 * i]),
                                            f.y + __uint_as_float(d[2 * i + 1]));
        out[i] = *reinterpret_cast<const uint32_t*>(&r);
      }
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
  }

  // ----------------------------------------------------------------------------- run ----
  // rank / n_tc: this CTA among the tensor CTAs.  n_mt: m-tiles of all long groups.
  __device__ __forceinline__ static void run(const Params& p, int S, uint8_t* smem,
                                             const int* starts, const int* adapters,
                                             const int* gcnt, const int* tbase, int* ctl,
                                             int rank, int n_tc, int n_mt) {
    const int tid = threadIdx.x, warp = tid >> 5;
    Ctx c;
    c.bars = smem_addr(smem + p.off_bars);
    c.ring = smem_addr(smem + p.tc_base);
    c.slots = p.tc_slots;
    c.rowtok = reinterpret_cast<int*>(smem + p.off_vpart);
    c.tmask = c.rowtok + 2 * kTcRows;
    c.starts = starts;
    c.adapters = adapters;
    c.gcnt = gcnt;
    c.tbase = tbase;
    c.S = S;
    c.xchg = smem_addr(smem + p.tc_xchg);
    // Split-K shrink over the 4 CTAs of a cluster (fused and shrink forms): member cr shrinks
    // chunks [nk cr / 4, nk (cr + 1) / 4) of h_in.
    c.split = kDoShrink ? 1 : 0;
    c.cr = c.split ? (rank & 3) : 0;
    {
      const int nk = kDoShrink ? (p.h_in + kTcK - 1) / kTcK : 0;
      c.k_lo = c.split ? nk * c.cr / 4 : 0;
      c.k_hi = c.split ? nk * (c.cr + 1) / 4 : nk;
    }
    uint32_t* tslot = reinterpret_cast<uint32_t*>(ctl + 1);
    if (tid == 0) {
      ctl[kCtlPending] = 0;
      ctl[kCtlTileGo] = -1;
      for (int s = 0; s < c.slots; ++s) {
        mbar_init(c.full(s), 32 + 1);  // the filling warp's cp.async arrivals + TMA bytes
        mbar_init(c.empty(s), 1 + 4);
      }
      mbar_init(c.fx(kTcVFull), 1);
      mbar_init(c.fx(kTcVFree), kTcEpi);
      mbar_init(c.fx(kTcHReady), kTcEpi);
      mbar_init(c.fx(kTcHFree), 1);
      mbar_init(c.fx(kTcDFull0), 1);
      mbar_init(c.fx(kTcDFull1), 1);
      mbar_init(c.fx(kTcDEmpty0), 4);
      mbar_init(c.fx(kTcDEmpty1), 4);
      mbar_init(c.fx(kTcRtFull0), 1);
      mbar_init(c.fx(kTcRtFull1), 1);
      mbar_init(c.fx(kTcRtFree0), kTcEpi * kGroups + 4);  // epilogue threads + 4 loader warps
      mbar_init(c.fx(kTcRtFree1), kTcEpi * kGroups + 4);
      mbar_init(c.fx(kTcRsFull), 1);  // the owner's expect_tx arrival + three partials' bytes
      mbar_init(c.fx(kTcAgFull), 1);  // the owner's expect_tx arrival + three owners' bytes
      mbar_init(c.fx(kTcNever), 1);
      mbar_init(c.fx(kTcDrain), 1);
      fence_mbar_init();
    }
    if (warp == kConsumerWarps) {
      tmem_alloc(smem_addr(tslot), kTcCols);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tslot;
    if (c.split) {  // every member's barriers exist before the first st.async (published by
      cluster_arrive_relaxed();  // the init fence above)
      cluster_wait();
    }

    if (tid == 0) {
      tma_prefetch_desc(&p.tmap_x128);
      tma_prefetch_desc(&p.tmap_x8);
      tma_prefetch_desc(&p.tmap_y128);
      tma_prefetch_desc(&p.tmap_y8);
    }
    const Waiter w{reinterpret_cast<volatile int*>(ctl), p.err, p.wait_limit_ns};
    if (p.inject_stall) w.wait<false>(c.fx(kTcNever), 0);  // nothing completes it

    TcWalk wk;
    wk.ntile = kDoExpand ? (p.h_out + kTcN - 1) / kTcN : 1;
    wk.split = c.split;
    wk.cr = c.cr;
    // Work units: clusters with the split-K shrink (all members walk the cluster's range),
    // single CTAs otherwise.
    const int unit = c.split ? rank >> 2 : rank;
    const int n_units = c.split ? n_tc >> 2 : n_tc;
    if (n_mt <= n_units && c.split) {
      // Fewer m-tiles than units: every m-tile gets the same k = floor(n_units / n_mt) units,
      // which split its n-tiles, so that no unit repeats a second shrink; the other units
      // idle.  Giving the remainder to some m-tiles cannot shorten the launch (the m-tiles
      // with k units still take as long) and adds their shrinks to the HBM traffic: measured
      // on the prefill mix (31 m-tiles, 36 clusters), 60.3 us with 5 m-tiles shared by two
      // clusters, 57.2 us with those 5 clusters idle.  (Without a shrink, a range that crosses
      // m-tiles costs one more read of v rows, so the expand-only form always takes the equal
      // contiguous ranges below: whole m-tiles per unit left 12 of 152 CTAs with 43 n-tiles
      // against 34-35 there.)
      const int k = n_units / n_mt;
      const int mi = unit / k, j = unit - mi * k;
      wk.u = mi < n_mt ? mi * wk.ntile + j * wk.ntile / k : 0;
      wk.u1 = mi < n_mt ? mi * wk.ntile + (j + 1) * wk.ntile / k : 0;
    } else {  // contiguous equal ranges of the (m-tile, n-tile) sequence
      const long long U = static_cast<long long>(n_mt) * wk.ntile;
      wk.u = static_cast<int>(U * unit / n_units);
      wk.u1 = static_cast<int>(U * (unit + 1) / n_units);
    }

    uint32_t filled = 0;  // loader warps: slots filled and their parities (drain)
    if (warp < 4) {
      filled = loader(p, c, w, wk);
    } else if (warp < kConsumerWarps) {
      epilogue(p, c, w, wk, tm, 0, ctl);
    } else if (kGroups == 2 && warp > kConsumerWarps) {
      epilogue(p, c, w, wk, tm, 1, ctl);
    } else if (warp == kConsumerWarps && (tid & 31) == 0) {
      issuer(p, c, w, wk, tm);
      // every MMA issued has completed before TMEM is released
      umma_commit(c.fx(kTcDrain));
      const uint64_t t0 = now_ns();
      while (!mbar_try(c.fx(kTcDrain), 0) && now_ns() - t0 < p.wait_limit_ns) {
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!w.ok()) {
      // Gave up: before the CTA exits, wait (bounded) for every asynchronous copy into its
      // shared memory -- the TMA loads of each slot's last fill (cp.async copies were waited
      // for by their warps) and the exchange data that peers may still be pushing.
      if (warp < 4 && (tid & 31) == 0)
        for (int s = 0; s < c.slots; ++s)
          if ((filled >> s) & 1u) w.drain<false>(c.full(s), (filled >> (16 + s)) & 1u);
      if (tid == 0 && ctl[kCtlPending]) {
        const uint32_t ph = static_cast<uint32_t>(ctl[kCtlPending] - 1);
        w.drain<true>(c.fx(kTcRsFull), ph);
        w.drain<true>(c.fx(kTcAgFull), ph);
      }
      __syncthreads();
    }
    if (warp == kConsumerWarps) tmem_dealloc(tm, kTcCols);
    if (c.split) {  // no member leaves while a peer may still write to it (every incoming
      cluster_arrive_relaxed();  // byte was counted by a barrier this CTA waited on)
      cluster_wait();
    }
  }
};

}  // namespace sgmv
