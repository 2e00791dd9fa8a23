// sgmv_core.cuh -- the segment scheduler and the CUDA-core shrink / expand / fused kernels.
//
// Operation (Punica Guide: Multi-Tenant LoRA Serving with SGMV; section "The Heterogeneous
// Batching Bottleneck", equation y_i = x_i W0 + (alpha/r) x_i A_k B_k; section "The SGMV
// Mathematical Formulation", segments [s_i, s_{i+1}) bound to one adapter each):
//     v[t]  = x[t] . A_k            shrink  (h_in -> r)
//     y[t] += scale * v[t] . B_k    expand  (r -> h_out)
//
// GB300 design (not the pages' Ampere design):
//  * Scheduler, in every CTA: the segment table is staged in shared memory and every segment
//    with an adapter is hashed by adapter id, so that all rows of one adapter -- even rows of
//    non-adjacent segments -- form one group whose weights are streamed once per call.  A
//    group is cut into work items of at most kRowsMax rows.  All CTAs derive the same item
//    list.  (The pages' "pre-sorted segment descriptors" and "one threadblock per segment",
//    section "Hardware-Level Optimizations in SGMV".)
//  * One item runs on a group of E CTAs (E = 1, 2 or 4, picked in the kernel from the item
//    count so that every SM has work; a group never spans two clusters).  Member m owns the
//    m-th slice of h_in (shrink, split-K) and of h_out (expand).
//  * Everything an item reads streams through one ring of shared-memory stages filled by 1-D
//    bulk copies (TMA) that one producer warp issues, in the order the consumers use it:
//    A-row chunks (each carrying the matching columns of the item's x rows), then per expand
//    pass the B-row chunks and one stage with the item's y rows.  Eight consumer warps compute
//    in fp32 on the CUDA cores.
//  * With E > 1 the r-wide partial products are summed through distributed shared memory in a
//    fixed member order (deterministic), so the intermediate v never leaves the cluster.
//  * Programmatic dependent launch: a kernel lets the next one start at once; the producer
//    fills the ring with weights, then waits for the previous kernel before any activation
//    copy (x, y, v).
//  * Groups with enough rows and weight re-use (a host-set row threshold) go to the tensor
//    role (sgmv_tc.cuh) on the first CTAs of the grid, whole clusters, in proportion to the
//    estimated bytes of each side; the other CTAs run the items above.
//  * Two instantiations per (type, rank, mode): 288 threads, two CTAs per SM (the default
//    geometry), and 416 threads, one CTA per SM (long batches of few segments; the extra
//    warps are a second tensor-role epilogue warpgroup and idle in the CUDA-core role).
//  * Every wait is bounded (globaltimer); a wait that runs out flags the CTA, sets the
//    library's device error word and lets the kernel run to its end without touching global
//    memory again.
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sgmv_ptx.cuh"

namespace sgmv {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp (two CTAs per SM)
// Long-batch launches (one CTA per SM): + four warps, a second tensor-role epilogue warpgroup.
constexpr int kThreadsWide = kThreads + 128;
constexpr int kStatusTimeout = -5;         // SGMV_ETIMEOUT
constexpr int kStatusBadPlan = -6;         // SGMV_EPLAN
constexpr int kPlanMagic = 0x504d4753;     // plan header word 0
constexpr int kPlanHeader = 16;            // ints before the group table
constexpr int kMaxProblems = 4;            // projections of one lora_apply_multi launch
constexpr int kRowsMax = 4;                // rows per CUDA-core work item

enum Mode : int { kFused = 0, kShrink = 1, kExpand = 2 };

// Barrier slots after the 2*nstages ring barriers.
enum Bar : int { kDescFull0 = 0, kDescFull1, kDescFree0, kDescFree1, kVReady0, kVReady1, kNever,
                 kNumFixedBars };

constexpr int kMaxGroup = 4;   // largest number of CTAs that share one item (launch cluster size)
constexpr int kPlanSlots = 7;  // member plans: E = 1 (slot 0), E = 2 (slots 1-2), E = 4 (3-6)

// What one member of a group of E CTAs streams for an item (computed on the host, so that the
// kernel does no division by runtime values).  Expand passes: all but the last cover w_full
// columns of the member's h_out slice, the last covers w_last; each pass is nb B chunks of cb
// B rows (the last chunk may be shorter) and one stage of y rows.
struct MemberPlan {
  int32_t k0, kc;        // h_in slice [k0, k0 + kc)
  int32_t nA, kbe;       // A chunks, A rows per chunk (a multiple of 8)
  int32_t n0, nc;        // h_out slice [n0, n0 + nc)
  int32_t passes;        // expand passes
  int32_t w_full, cb_full, nb_full;
  int32_t w_last, cb_last, nb_last;
  int32_t total;         // ring stages per item
};

// A CUDA tensor map (the driver's 128-byte opaque descriptor), 64-byte aligned as TMA needs.
struct alignas(64) TmaMap {
  uint64_t q[16];
};

struct Params {
  void* y;
  const void* x;
  float* v_out;
  const float* v_in;
  const void* const* A_ptrs;
  const void* const* B_ptrs;
  const int32_t* seg_starts;
  const int32_t* seg_adapter;
  int* err;  // library device error word
  int32_t S, layer, h_in, h_out;
  int32_t ldx, ldy;     // row strides of x and y, in elements (>= h_in / h_out)
  float scale;
  int32_t C;            // launch cluster size (a multiple of every group size used)
  int32_t nstages;      // ring stages
  int32_t stage_bytes;  // bytes per ring stage
  int32_t kb;           // x-row stride (elements) inside an A stage (>= every kbe)
  int32_t hash_slots;   // power of two > 1.5*S
  uint32_t off_bars, off_ctl, off_desc, off_tab, off_vpart, off_vfull, off_red, off_stab,
      off_ring;
  int32_t desc_ints;
  uint64_t wait_limit_ns;
  int32_t inject_stall;
  // Launched as a programmatic dependent of the previous kernel (SGMV_OVERLAP_PRIOR): the
  // activations may only be read after griddepcontrol.wait.  Otherwise the previous kernel has
  // completed before this one started and they are copied with the weights from the start.
  int32_t dependent;
  int32_t tc_min_rows;  // groups with at least this many rows go to the tensor role (INT32_MAX: none)
  int32_t tc_slots;     // tensor-role ring slots (24 KB each)
  uint32_t tc_base;     // tensor-role ring offset (1024-aligned; after its row table at off_vpart)
  uint32_t tc_xchg;     // tensor-role split-K exchange buffers (after the ring)
  int32_t xchg_bytes;   // cost of one partial-sum exchange, in streamed bytes (group size rule)
  MemberPlan plan[kPlanSlots];
  // A plan built by sgmv_plan (nullptr: the segment table is grouped by every CTA).  With a
  // plan, seg_starts / seg_adapter point at its group table (one segment per adapter group,
  // S = capacity, the group count in the plan header) and the rows of group segment g are
  // rowmap[seg_starts[g] .. seg_starts[g + 1]).
  const int32_t* plan_hdr;
  const int32_t* rowmap;
  // Per-adapter rank and scale (lora_apply_ranked; nullptr: every adapter has rank R and
  // `scale`).  Adapter k's blocks are [L][h_in][r_k] and [L][r_k][h_out] (rank_of).  The
  // kernels keep R (the call's r_max) as their capacity: columns of v past r_k stay exactly
  // zero and B rows past r_k are never read.
  const int32_t* adapter_rank;
  const float* adapter_scale;
  int32_t cta0, nctas;  // this problem's CTAs in the grid (a multiple of C)
  // Tensor role: x [rows][h_in] and y [rows][h_out] with the 128-byte swizzle, boxes of
  // 64 elements x 128 rows (a whole m-tile) and 64 x 8 rows (one swizzle atom).
  TmaMap tmap_x128, tmap_x8, tmap_y128, tmap_y8;
  // ... and 64 x 64 / 32 / 16 rows, for a tile whose rows are one shorter run (segment ends).
  TmaMap tmap_x64, tmap_x32, tmap_x16, tmap_y64, tmap_y32, tmap_y16;
};

// ---- element types ---------------------------------------------------------------------
template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16 bytes
  __device__ static __forceinline__ void lds(uint32_t a, float (&o)[4]) {
    const uint4 v = lds128(a);
    o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ float lds1(uint32_t a) { return __uint_as_float(lds32(a)); }
  __device__ static __forceinline__ void sts(uint32_t a, const float (&o)[4]) {
    sts128(a, make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                         __float_as_uint(o[3])));
  }
  __device__ static __forceinline__ void load16(const void* p, float (&o)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  __device__ static __forceinline__ float load1(const void* p) {
    return *reinterpret_cast<const float*>(p);
  }
  __device__ static __forceinline__ void store16(void* p, const float (&o)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};
template <>
struct Elem<__half> {
  static constexpr int kVec = 8;
  // acc += a * b with a, b fp16 bit patterns: the product is exact in fp32, so this equals
  // converting both to fp32 first and using fmaf (one instruction instead of three).
  __device__ static __forceinline__ void fma16(float& acc, uint16_t a, uint16_t b) {
    asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(b));
  }
  __device__ static __forceinline__ void lds(uint32_t a, float (&o)[8]) {
    const uint4 v = lds128(a);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    }
  }
  __device__ static __forceinline__ float lds1(uint32_t a) {
    const unsigned short h = static_cast<unsigned short>(lds16(a));
    return __half2float(*reinterpret_cast<const __half*>(&h));
  }
  __device__ static __forceinline__ void sts(uint32_t a, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    sts128(a, make_uint4(w[0], w[1], w[2], w[3]));
  }
  __device__ static __forceinline__ void load16(const void* p, float (&o)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    }
  }
  __device__ static __forceinline__ float load1(const void* p) {
    return __half2float(*reinterpret_cast<const __half*>(p));
  }
  __device__ static __forceinline__ void store16(void* p, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static __forceinline__ void fma16(float& acc, uint16_t a, uint16_t b) {
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(b));
  }
  __device__ static __forceinline__ void lds(uint32_t a, float (&o)[8]) {
    const uint4 v = lds128(a);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // bf16 -> fp32 is exact: the bf16 bits are the high half
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static __forceinline__ float lds1(uint32_t a) {
    return __uint_as_float(lds16(a) << 16);
  }
  __device__ static __forceinline__ void sts(uint32_t a, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    sts128(a, make_uint4(w[0], w[1], w[2], w[3]));
  }
  __device__ static __forceinline__ void load16(const void* p, float (&o)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // bf16 -> fp32 is exact: the bf16 bits are the high half
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static __forceinline__ float load1(const void* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
  __device__ static __forceinline__ void store16(void* p, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// ---- bounded waits ----------------------------------------------------------------------
struct Waiter {
  volatile int* abort;  // CTA-wide flag in shared memory
  int* err;
  uint64_t limit;

  // Returns false (without waiting) once the CTA has given up, or when the bound runs out.
  template <bool kCluster>
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    if (*abort) return false;
    if (kCluster ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (true) {
#pragma unroll 1
      for (int i = 0; i < 8; ++i)
        if (kCluster ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
      if (*abort) return false;
      if (now_ns() - t0 > limit) {
        *abort = 1;
        atomicExch(err, kStatusTimeout);
        return false;
      }
    }
  }
  __device__ __forceinline__ bool ok() const { return *abort == 0; }

  // Bounded wait until the shared counter *f reaches `target` (a monotonic counter cannot alias
  // the way an mbarrier parity can).  All threads that call it see the same result only if
  // the caller makes them agree (e.g. __all_sync).
  __device__ __forceinline__ bool until(const volatile int* f, int target) const {
    if (*f >= target) return true;
    const uint64_t t0 = now_ns();
    while (true) {
      if (*f >= target) return true;
      if (*abort) return false;
      if (now_ns() - t0 > limit) {
        *abort = 1;
        atomicExch(err, kStatusTimeout);
        return false;
      }
    }
  }

  // After the CTA gave up: waits (bounded, ignoring the abort flag) until the phase of `bar`
  // with this parity has completed, i.e. until the asynchronous copies counted on it have
  // landed in this CTA's shared memory.  Returns false when the bound ran out (copies whose
  // bytes were announced but never issued).
  template <bool kCluster>
  __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
    const uint64_t t0 = now_ns();
    while (!(kCluster ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)))
      if (now_ns() - t0 > limit) return false;
    return true;
  }
};

// Shared-memory control words (ints at off_ctl): [0] abort flag, [1] TMEM address (tensor
// role), [2..3] tensor_ctas sums, [4..23] scan scratch, and the drain records below.
constexpr int kCtlIssued = 26;   // ring slots the producer ever filled (bit mask)
constexpr int kCtlParity = 27;   // phase parity of each slot's last fill (bit mask)
constexpr int kCtlPending = 28;  // 1 + parity of an armed exchange barrier not yet seen complete
constexpr int kCtlPendBar = 29;  // which exchange barrier
constexpr int kCtlTileGo = 30;   // tensor role: last m-tile whose shrink slots are all consumed

// ---- stage layout ---------------------------------------------------------------------
// The stages of one item, in ring order: [A chunks][pass 0: B chunks, y][pass 1: ...] (fused);
// [A chunks] (shrink); [v][pass 0: B chunks, y]... (expand).
enum ChunkKind : int { kChunkA = 0, kChunkB = 1, kChunkY = 2, kChunkV = 3, kChunkEnd = 4 };

static __device__ __forceinline__ int b_row_stride(int w, int eb) { return w * eb + 16; }

// Walks the stages of an item in ring order (increments only, no division).
template <int R, int MODE>
struct StageWalk {
  int kind, a, pass, c0, rows, wdt, cb;
  __device__ __forceinline__ void set_pass(const MemberPlan& mp, int ps) {
    pass = ps;
    const bool lastp = ps == mp.passes - 1;
    wdt = lastp ? mp.w_last : mp.w_full;
    cb = lastp ? mp.cb_last : mp.cb_full;
    kind = kChunkB;
    c0 = 0;
    rows = min(cb, R);
  }
  __device__ __forceinline__ void after_a(const MemberPlan& mp) {
    if (MODE != kShrink && mp.passes > 0) set_pass(mp, 0); else kind = kChunkEnd;
  }
  __device__ __forceinline__ void first(const MemberPlan& mp) {
    a = 0;
    pass = 0;
    c0 = 0;
    wdt = 0;
    cb = 0;
    if (MODE == kExpand) {
      kind = kChunkV;
    } else if (mp.nA > 0) {
      kind = kChunkA;
      rows = min(mp.kbe, mp.kc);
    } else {
      after_a(mp);
    }
  }
  __device__ __forceinline__ void next(const MemberPlan& mp) {
    if (kind == kChunkV) {
      after_a(mp);
    } else if (kind == kChunkA) {
      if (++a < mp.nA) rows = min(mp.kbe, mp.kc - a * mp.kbe); else after_a(mp);
    } else if (kind == kChunkB) {
      c0 += cb;
      if (c0 < R) rows = min(cb, R - c0); else kind = kChunkY;
    } else if (kind == kChunkY) {
      if (pass + 1 < mp.passes) set_pass(mp, pass + 1); else kind = kChunkEnd;
    }
  }
};

// Ring slot iterator: slot s, phase parity of the current round, whether a round completed.
struct RingPos {
  int s;
  uint32_t par;
  bool wrapped;
  __device__ __forceinline__ void init() {
    s = 0;
    par = 0;
    wrapped = false;
  }
  __device__ __forceinline__ void next(int nst) {
    if (++s == nst) {
      s = 0;
      par ^= 1u;
      wrapped = true;
    }
  }
};

// ---- scheduler ------------------------------------------------------------------------
// Exclusive scan of `cnt(i)` over i in [0, n) into out[0..n] (out[n] = total), all threads.
template <int NT, typename F>
__device__ __forceinline__ void block_exclusive_scan(int n, int* out, int* wsum, F cnt) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = NT / 32;
  const int per = (n + NT - 1) / NT;
  const int lo = min(tid * per, n), hi = min(lo + per, n);
  int local = 0;
  for (int i = lo; i < hi; ++i) local += cnt(i);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int v = wsum[w];
      wsum[w] = run;
      run += v;
    }
    wsum[kWarps] = run;
  }
  __syncthreads();
  int off = wsum[warp] + incl - local;
  for (int i = lo; i < hi; ++i) {
    out[i] = off;
    off += cnt(i);
  }
  if (tid == 0) out[n] = wsum[kWarps];
  __syncthreads();
}

static __device__ __forceinline__ uint32_t hash_slot(int k, int mask) {
  return ((static_cast<uint32_t>(k) * 0x9E3779B1u) >> 12) & static_cast<uint32_t>(mask);
}

// Builds, in shared memory: starts[0..S], adapters[0..S-1], base[0..S] where base is the
// exclusive prefix of "work items led by segment i".  Segment i leads its group when it is the
// first non-empty segment of its adapter; its group gets ceil(rows / kRowsMax) items, and
// gcnt[lead] holds the group's row count.
// `scratch` (transient) holds slot[S] and the hash table (3 * hash_slots ints).
template <int NT>
static __device__ __forceinline__ void build_schedule(const Params& p, int S, int* starts,
                                                      int* adapters, int* base, int* gcnt,
                                                      int* tbase, int* scratch, int* wsum) {
  const int tid = threadIdx.x;
  const int HS = p.hash_slots;
  int* slot = scratch;
  int* hkey = slot + S;
  int* hlead = hkey + HS;
  int* hcnt = hlead + HS;
  // Table loads go out first (registers), the hash is cleared while they are in flight.
  constexpr int kPer = 4;
  int st_v[kPer], ad_v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * NT;
    st_v[u] = (i <= S) ? __ldg(p.seg_starts + i) : 0;
    ad_v[u] = (i < S) ? __ldg(p.seg_adapter + i) : 0;
  }
  for (int h = tid; h < HS; h += NT) {
    hkey[h] = -1;
    hlead[h] = 0x7fffffff;
    hcnt[h] = 0;
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * NT;
    if (i <= S) starts[i] = st_v[u];
    if (i < S) adapters[i] = ad_v[u];
  }
  for (int i = tid + kPer * NT; i <= S; i += NT) {
    starts[i] = __ldg(p.seg_starts + i);
    if (i < S) adapters[i] = __ldg(p.seg_adapter + i);
  }
  __syncthreads();
  // A plan's group table is already grouped: every segment is its own group's lead.
  if (p.plan_hdr) {
    for (int i = tid; i < S; i += NT) {
      slot[i] = i;
      hlead[i] = i;
      hcnt[i] = starts[i + 1] - starts[i];
    }
  }
  for (int i = tid; i < S && !p.plan_hdr; i += NT) {
    const int k = adapters[i];
    const int len = starts[i + 1] - starts[i];
    int h = -1;
    if (k >= 0 && len > 0) {
      h = static_cast<int>(hash_slot(k, HS - 1));
      while (true) {  // at most S distinct keys in HS > 1.5 S slots: terminates
        const int prev = atomicCAS(&hkey[h], -1, k);
        if (prev == -1 || prev == k) break;
        h = (h + 1) & (HS - 1);
      }
      atomicMin(&hlead[h], i);
      atomicAdd(&hcnt[h], len);
    }
    slot[i] = h;
  }
  __syncthreads();
  const int tcmin = p.tc_min_rows;
  int* any_long = wsum + NT / 32 + 1;  // set when some group goes to the tensor role
  if (threadIdx.x == 0) *any_long = 0;
  block_exclusive_scan<NT>(S, base, wsum, [&](int i) {
    const int h = slot[i];
    const bool lead = h >= 0 && hlead[h] == i;
    const int rows = lead ? hcnt[h] : 0;
    gcnt[i] = rows;
    if (rows >= tcmin) *any_long = 1;
    return rows >= tcmin ? 0 : (rows + kRowsMax - 1) / kRowsMax;
  });
  // Groups of at least tc_min_rows rows: m-tiles of 128 rows for the tensor role.
  if (*any_long)
    block_exclusive_scan<NT>(S, tbase, wsum, [&](int i) {
      const int rows = gcnt[i];
      return rows >= tcmin ? (rows + 127) / 128 : 0;
    });
  else if (threadIdx.x == 0)
    tbase[S] = 0;
  __syncthreads();
}

// Rank of adapter k: R in an unranked call; in a ranked call its entry when that is a multiple
// of 8 in [8, R], else 0 -- the adapter is then skipped (its rows get exactly + 0), so that no
// entry can make the kernel read past the block size the caller declared.
template <int R>
static __device__ __forceinline__ int rank_of(const Params& p, int k) {
  if (!p.adapter_rank) return R;
  const int v = __ldg(p.adapter_rank + k);
  return (v >= 8 && v <= R && (v & 7) == 0) ? v : 0;
}
static __device__ __forceinline__ float scale_of(const Params& p, int k) {
  return p.adapter_scale ? __ldg(p.adapter_scale + k) : p.scale;
}

// Token index of (virtual) row v: with a plan, rows are listed group by group in its row map.
static __device__ __forceinline__ int row_of(const Params& p, int v) {
  return p.rowmap ? __ldg(p.rowmap + v) : v;
}

// One warp: turns item t into {adapter, rows, row ids...} in d (d[0]=k, d[1]=R, d[2..]=rows).
static __device__ __forceinline__ void decode_item(const Params& p, int S, int t,
                                                   const int* starts, const int* adapters,
                                                   const int* base, const int* gcnt, int* d) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = S - 1;  // largest i with base[i] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int lead = lo;
  const int k = adapters[lead];
  const int p_lo = (t - base[lead]) * kRowsMax;
  const int p_hi = min(p_lo + kRowsMax, gcnt[lead]);  // stop once the chunk's rows are found
  if (p.rowmap) {  // a plan's group is one segment: its rows are consecutive in the row map
    if (lane < p_hi - p_lo) d[2 + lane] = __ldg(p.rowmap + starts[lead] + p_lo + lane);
    if (lane == 0) {
      d[0] = k;
      d[1] = max(0, p_hi - p_lo);
    }
    __syncwarp();
    return;
  }
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
    const int a = max(seg_lo, p_lo), b = min(pos + incl, p_hi);
    for (int q = a; q < b; ++q) d[2 + q - p_lo] = row_of(p, starts[j] + (q - seg_lo));
    pos += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    d[0] = k;
    d[1] = max(0, min(pos, p_hi) - p_lo);
  }
  __syncwarp();
}

}  // namespace sgmv

#include "sgmv_tc.cuh"

namespace sgmv {

// ---- the kernel ------------------------------------------------------------------------
template <typename T, int R, int MODE, int NT>
struct Kernel {
  using E = Elem<T>;
  using Walk = StageWalk<R, MODE>;
  static constexpr int kVec = E::kVec;
  static constexpr int kCpr = R / kVec;  // 16-byte chunks per A row
  static constexpr int kKLanes = kConsumers / kCpr;
  static constexpr int kEb = sizeof(T);
  static_assert(kCpr >= 1 && kCpr <= 32, "rank / vector width");

  // Shared-memory map with every address precomputed once per CTA.
  struct Smem {
    uint32_t bars_u32;  // barrier 0
    uint8_t* ring;      // stage 0
    uint32_t ring_u32;
    int nst, stage_bytes, desc_ints;
    int* desc_p;
    float *vpart_p, *vfull_p, *red_p;
    __device__ __forceinline__ void init(uint8_t* smem, const Params& p) {
      bars_u32 = smem_addr(smem + p.off_bars);
      ring = smem + p.off_ring;
      ring_u32 = smem_addr(ring);
      nst = p.nstages;
      stage_bytes = p.stage_bytes;
      desc_ints = p.desc_ints;
      desc_p = reinterpret_cast<int*>(smem + p.off_desc);
      vpart_p = reinterpret_cast<float*>(smem + p.off_vpart);
      vfull_p = reinterpret_cast<float*>(smem + p.off_vfull);
      red_p = reinterpret_cast<float*>(smem + p.off_red);
    }
    __device__ __forceinline__ uint32_t bar(int i) const {
      return bars_u32 + 8u * static_cast<uint32_t>(i);
    }
    __device__ __forceinline__ uint32_t full(int s) const { return bar(s); }
    __device__ __forceinline__ uint32_t empty(int s) const { return bar(nst + s); }
    __device__ __forceinline__ uint32_t fixed(int b) const { return bar(2 * nst + b); }
    __device__ __forceinline__ uint8_t* stage(int s) const {
      return ring + static_cast<uint32_t>(s) * static_cast<uint32_t>(stage_bytes);
    }
    __device__ __forceinline__ uint32_t stage_u32(int s) const {
      return ring_u32 + static_cast<uint32_t>(s) * static_cast<uint32_t>(stage_bytes);
    }
    __device__ __forceinline__ int* desc(int b) const { return desc_p + b * desc_ints; }
    // partial products of member m for item parity b: [2][kMaxGroup][kRowsMax][R]
    __device__ __forceinline__ float* vpart(int b, int m) const {
      return vpart_p + (b * kMaxGroup + m) * kRowsMax * R;
    }
  };

  // The CTAs that share one item.
  struct Group {
    int size;     // E
    int m;        // this CTA's member index
    int gid, ng;  // group index, number of groups
    int rank0;    // cluster rank of member 0
  };

  // ------------------------------------------------------------------ producer warp ----
  // Stage descriptors of one item: {kind | rows << 4, offset, column, width}.  A: offset = first
  // h_in element of the chunk; B: offset = first B row, column = first h_out column, width =
  // window width; Y: column, width.  Built by the 32 producer lanes in parallel so that the issue
  // loop is a few instructions per stage.
  __device__ __forceinline__ static void build_table(const MemberPlan& mp, int4* tab) {
    const int lane = threadIdx.x & 31;
    for (int t = lane; t < mp.total; t += 32) {
      int u = t;
      int4 e = make_int4(kChunkV, 0, 0, 0);
      if (MODE == kExpand) --u;
      if (u >= 0) {
        if (u < mp.nA) {
          const int rows = min(mp.kbe, mp.kc - u * mp.kbe);
          e = make_int4(kChunkA | (rows << 4), mp.k0 + u * mp.kbe, 0, 0);
        } else {
          u -= mp.nA;
          const int per = mp.nb_full + 1, nfull = mp.passes - 1;
          int pass, jj, w, cb, nb;
          if (u < nfull * per) {
            pass = u / per;
            jj = u - pass * per;
            w = mp.w_full;
            cb = mp.cb_full;
            nb = mp.nb_full;
          } else {
            pass = nfull;
            jj = u - nfull * per;
            w = mp.w_last;
            cb = mp.cb_last;
            nb = mp.nb_last;
          }
          const int col = mp.n0 + pass * mp.w_full;
          if (jj < nb) {
            const int c0 = jj * cb;
            e = make_int4(kChunkB | (min(cb, R - c0) << 4), c0, col, w);
          } else {
            e = make_int4(kChunkY, 0, col, w);
          }
        }
      }
      tab[t] = e;
    }
    __syncwarp();
  }

  // Activation part of a stage (x columns of an A chunk, y rows of a pass, v rows) into slot s.
  __device__ __forceinline__ static void issue_acts(const Params& p, const Smem& sm, bool ok,
                                                    int4 e, int s, const int* d, int nrow,
                                                    uint64_t pol) {
    const int lane = threadIdx.x & 31;
    if (!ok || lane >= nrow) return;
    const int kind = e.x & 15;
    const int row = d[2 + lane];
    if (kind == kChunkA) {
      const int rows = e.x >> 4;
      bulk_g2s(sm.stage_u32(s) + static_cast<uint32_t>((p.kb * R + lane * p.kb) * kEb),
               static_cast<const T*>(p.x) + static_cast<size_t>(row) * p.ldx + e.y,
               static_cast<uint32_t>(rows * kEb), sm.full(s), pol);
    } else if (kind == kChunkY) {
      bulk_g2s(sm.stage_u32(s) + static_cast<uint32_t>(lane * e.w * kEb),
               static_cast<const T*>(p.y) + static_cast<size_t>(row) * p.ldy + e.z,
               static_cast<uint32_t>(e.w * kEb), sm.full(s), pol);
    } else if (kind == kChunkV) {
      bulk_g2s(sm.stage_u32(s) + static_cast<uint32_t>(lane * R * 4),
               p.v_in + static_cast<size_t>(row) * R, R * 4, sm.full(s), pol);
    }
  }

  // One stage into the current ring slot: wait for the slot (after the first round), announce
  // its bytes (weights and activations), copy the weights, and the activations when `acts`.
  // Returns whether the stage's bytes were announced (false once the CTA has given up).  rk:
  // the item's adapter rank (A rows are rk elements; B rows past rk are not copied).
  __device__ __forceinline__ static bool issue_stage(const Params& p, const Smem& sm,
                                                     const Waiter& w, int4 e, const RingPos& rp,
                                                     const T* Ak, const T* Bk, const int* d,
                                                     int nrow, bool acts, uint64_t pol_w,
                                                     uint64_t pol_a, int rk) {
    const int lane = threadIdx.x & 31;
    const int s = rp.s;
    const int kind = e.x & 15;
    const int rows = kind == kChunkB ? max(0, min(e.x >> 4, rk - e.y)) : (e.x >> 4);
    if (lane == 0) {
      if (rp.wrapped) w.wait<false>(sm.empty(s), rp.par ^ 1u);
      const bool ok = w.ok();
      uint32_t bytes;
      if (kind == kChunkA)
        bytes = static_cast<uint32_t>((rk + nrow) * rows * kEb);
      else if (kind == kChunkB)
        bytes = static_cast<uint32_t>(rows * e.w * kEb);
      else if (kind == kChunkY)
        bytes = static_cast<uint32_t>(nrow * e.w * kEb);
      else
        bytes = static_cast<uint32_t>(nrow * R * 4);
      mbar_arrive_expect_tx(sm.full(s), ok ? bytes : 0u);
      if (kind == kChunkA && ok && rk > 0)
        bulk_g2s(sm.stage_u32(s), Ak + static_cast<size_t>(e.y) * rk,
                 static_cast<uint32_t>(rows * rk * kEb), sm.full(s), pol_w);
    }
    // every lane follows lane 0's decision, so that the bytes announced are the bytes copied
    const bool ok = __shfl_sync(0xffffffffu, w.ok() ? 1 : 0, 0) != 0;
    if (kind == kChunkB && ok)
      for (int rr = lane; rr < rows; rr += 32)  // up to R (64) rows
        bulk_g2s(sm.stage_u32(s) + static_cast<uint32_t>(rr * b_row_stride(e.w, kEb)),
                 Bk + static_cast<size_t>(e.y + rr) * p.h_out + e.z,
                 static_cast<uint32_t>(e.w * kEb), sm.full(s), pol_w);
    if (acts) issue_acts(p, sm, ok, e, s, d, nrow, pol_a);
    return ok;
  }

  __device__ __forceinline__ static void producer(const Params& p, const Smem& sm,
                                                  const Waiter& w, const Group& grp,
                                                  const MemberPlan& mp, const int* starts,
                                                  const int* adapters, const int* base,
                                                  const int* gcnt, int4* tab, int n_my,
                                                  int* ctl, int S) {
    const int lane = threadIdx.x & 31;
    uint32_t issued = 0, parity = 0;  // ring slots filled, parity of each one's last fill
    uint32_t pre_ok = 0;  // stages issued before the wait on the previous kernel, bytes announced
    const uint64_t pol_w = policy_evict_first();  // weights: streamed once per call
    const uint64_t pol_a = policy_evict_last();   // activations: reused by the group
    const int NST = sm.nst;
    const int total = mp.total;
    RingPos rp;
    rp.init();
    bool prior_done = !p.dependent;  // nothing to wait for: activations go with their stages
    for (int li = 0; li < n_my; ++li) {
      const int b = li & 1;
      if (li >= 2 && lane == 0) w.wait<false>(sm.fixed(kDescFree0 + b), ((li >> 1) - 1) & 1);
      __syncwarp();
      int* d = sm.desc(b);
      decode_item(p, S, grp.gid + li * grp.ng, starts, adapters, base, gcnt, d);
      if (lane == 0) {  // the adapter's rank and scale travel with the item
        d[6] = rank_of<R>(p, d[0]);
        d[7] = __float_as_int(scale_of(p, d[0]));
        mbar_arrive(sm.fixed(kDescFull0 + b));
      }
      __syncwarp();
      const int k = d[0];
      const int rk = d[6];
      const int nrow = min(max(d[1], 0), kRowsMax);
      const T* Ak = nullptr;
      const T* Bk = nullptr;
      if (MODE != kExpand)
        Ak = static_cast<const T*>(p.A_ptrs[k]) + static_cast<size_t>(p.layer) * p.h_in * rk;
      if (MODE != kShrink)
        Bk = static_cast<const T*>(p.B_ptrs[k]) + static_cast<size_t>(p.layer) * rk * p.h_out;
      if (li == 0) build_table(mp, tab);  // the plan is the same for every item of this CTA
      for (int t = 0; t < total; ++t, rp.next(NST)) {
        if (!prior_done && rp.wrapped) {
          // The ring is full of weights, which do not depend on the previous kernel of the
          // stream; before a slot is reused, wait for that kernel and add the activations of
          // the stages already issued (item 0 started at slot 0).
          pdl_wait_prior();
          prior_done = true;
          // the activation bytes of a stage were announced with its weights (or none were):
          // copy exactly what was announced, so that every phase completes
          for (int q = 0; q < t; ++q)
            issue_acts(p, sm, (pre_ok >> q) & 1u, tab[q], q, d, nrow, pol_a);
        }
        const bool sok = issue_stage(p, sm, w, tab[t], rp, Ak, Bk, d, nrow, prior_done, pol_w,
                                     pol_a, rk);
        if (!prior_done && sok) pre_ok |= 1u << t;
        issued |= 1u << rp.s;
        parity = (parity & ~(1u << rp.s)) | (rp.par << rp.s);
      }
      if (!prior_done) {
        pdl_wait_prior();
        prior_done = true;
        for (int q = 0; q < total; ++q)
          issue_acts(p, sm, (pre_ok >> q) & 1u, tab[q], q, d, nrow, pol_a);
      }
    }
    if (!prior_done) pdl_wait_prior();
    if (lane == 0) {  // for the drain of a CTA that gives up
      ctl[kCtlIssued] = static_cast<int>(issued);
      ctl[kCtlParity] = static_cast<int>(parity);
    }
  }

  // --------------------------------------------------------------- consumer warps ----
  // kRanked: the call has per-adapter ranks (rk read from the descriptor); otherwise rk is the
  // compile-time R, so that the hot loops keep constant strides.
  template <int RB, bool kRanked>
  __device__ __forceinline__ static void consume_item(const Params& p, const Smem& sm,
                                                      const Waiter& w, const Group& grp,
                                                      const MemberPlan& mp, int li, bool last,
                                                      RingPos& rp, const int* d, int nrow,
                                                      int* ctl) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NST = sm.nst;
    // The item's adapter rank (R unless ranked) and the scale of its term.  Clamped like nrow:
    // a CTA that has given up no longer waits for the descriptor, and whatever it then reads
    // must still index inside its own stages.
    const int rk = kRanked ? min(max(d[6], 0), R) & ~7 : R;
    const float sk = __int_as_float(d[7]);
    float acc[RB][kVec];
    float* vfull = sm.vfull_p;
    const uint32_t vfull_u32 = smem_addr(vfull);

    if (MODE == kExpand) {
      // ------------------------------------------------------------- v rows of the item
      w.wait<false>(sm.full(rp.s), rp.par);
      const float* vs = reinterpret_cast<const float*>(sm.stage(rp.s));
      for (int t = tid; t < nrow * R; t += kConsumers) vfull[t] = sk * vs[t];
      named_bar(1, kConsumers);
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty(rp.s));
      rp.next(NST);
    } else {
      // ----------------------------------------------------------- shrink (split-K)
#pragma unroll
      for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int e = 0; e < kVec; ++e) acc[i][e] = 0.f;
      const int cc = tid % kCpr, kl = tid / kCpr;  // compile-time divisors
      const bool col_ok = cc * kVec < rk;          // columns past the rank read as zero
      const int xrow = p.kb * kEb;
      const int xoff = p.kb * R * kEb;
      int rows = min(mp.kbe, mp.kc);
      for (int j = 0; j < mp.nA; ++j, rp.next(NST), rows = min(mp.kbe, mp.kc - j * mp.kbe)) {
        w.wait<false>(sm.full(rp.s), rp.par);
        const uint32_t st = sm.stage_u32(rp.s);
        const uint32_t xs = st + xoff;
        constexpr int U = RB <= 2 ? 4 : 2;  // rows in flight per thread (loads before FMAs)
        if constexpr (sizeof(T) == 2) {  // 16-bit operands straight into fp32 FMAs
          for (int kk0 = kl; kk0 < rows; kk0 += U * kKLanes) {
            uint4 a[U];
            uint16_t xv[U][RB];
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int kk = kk0 + u * kKLanes;
              if (kk < rows) {
                a[u] = col_ok ? lds128(st + (kk * rk + cc * kVec) * kEb)
                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int i = 0; i < RB; ++i)
                  xv[u][i] = static_cast<uint16_t>(lds16(xs + i * xrow + kk * kEb));
              } else {
                a[u] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int i = 0; i < RB; ++i) xv[u][i] = 0;
              }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const uint32_t wd[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
#pragma unroll
              for (int i = 0; i < RB; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  E::fma16(acc[i][2 * e], xv[u][i], static_cast<uint16_t>(wd[e] & 0xffffu));
                  E::fma16(acc[i][2 * e + 1], xv[u][i], static_cast<uint16_t>(wd[e] >> 16));
                }
            }
          }
        } else
        for (int kk0 = kl; kk0 < rows; kk0 += U * kKLanes) {
          float a[U][kVec], xv[U][RB];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int kk = kk0 + u * kKLanes;
            if (kk < rows && col_ok) {
              E::lds(st + (kk * rk + cc * kVec) * kEb, a[u]);
#pragma unroll
              for (int i = 0; i < RB; ++i) xv[u][i] = E::lds1(xs + i * xrow + kk * kEb);
            } else if (kk < rows) {
#pragma unroll
              for (int e = 0; e < kVec; ++e) a[u][e] = 0.f;
#pragma unroll
              for (int i = 0; i < RB; ++i) xv[u][i] = E::lds1(xs + i * xrow + kk * kEb);
            } else {
#pragma unroll
              for (int e = 0; e < kVec; ++e) a[u][e] = 0.f;
#pragma unroll
              for (int i = 0; i < RB; ++i) xv[u][i] = 0.f;
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < RB; ++i)
#pragma unroll
              for (int e = 0; e < kVec; ++e) acc[i][e] = fmaf(xv[u][i], a[u][e], acc[i][e]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty(rp.s));
      }
      // reduce over the k-lanes of the warp (lanes with equal cc), then over warps
#pragma unroll
      for (int o = kCpr; o < 32; o <<= 1)
#pragma unroll
        for (int i = 0; i < RB; ++i)
#pragma unroll
          for (int e = 0; e < kVec; ++e) acc[i][e] += __shfl_xor_sync(0xffffffffu, acc[i][e], o);
      float* red = sm.red_p;
      if (lane < kCpr) {
#pragma unroll
        for (int i = 0; i < RB; ++i)
#pragma unroll
          for (int e = 0; e < kVec; ++e)
            red[(warp * kRowsMax + i) * R + lane * kVec + e] = acc[i][e];
      }
      named_bar(1, kConsumers);
      if (grp.size == 1) {
        for (int t = tid; t < nrow * R; t += kConsumers) {
          float s = 0.f;
#pragma unroll
          for (int ww = 0; ww < kConsumerWarps; ++ww) s += red[ww * kRowsMax * R + t];
          if (MODE == kFused) {
            vfull[t] = s * sk;
          } else if (w.ok()) {
            p.v_out[static_cast<size_t>(d[2 + t / R]) * R + (t % R)] = s;
          }
        }
        named_bar(1, kConsumers);
      } else {
        // ------------------------------------------------- group all-reduce of v (DSMEM)
        // Every member pushes its partial into slot m of every member's buffer with
        // asynchronous stores that count bytes on that member's barrier; a member's barrier
        // completes once all E partials have landed, and the member sums the slots locally in
        // member order (deterministic).
        if (li == 0) cluster_wait();  // peers' barriers are initialised (arrive #1)
        const uint32_t vready = sm.fixed(kVReady0 + (li & 1));
        if (tid == 0)
          mbar_arrive_expect_tx(vready, static_cast<uint32_t>(grp.size * nrow * R * 4));
        const uint32_t my_slot = smem_addr(sm.vpart(li & 1, grp.m));
        for (int t = tid; t < nrow * R; t += kConsumers) {
          float s = 0.f;
#pragma unroll
          for (int ww = 0; ww < kConsumerWarps; ++ww) s += red[ww * kRowsMax * R + t];
          for (int j = 0; j < grp.size; ++j)
            st_async_f32(cluster_map(my_slot + 4u * t, grp.rank0 + j), s,
                         cluster_map(vready, grp.rank0 + j));
        }
        const bool got = w.wait<true>(vready, (li >> 1) & 1);
        if (tid == 0 && !got) {  // peers' pushes may still land: drained before exit
          ctl[kCtlPending] = 1 + ((li >> 1) & 1);
          ctl[kCtlPendBar] = kVReady0 + (li & 1);
        }
        for (int t = tid; t < nrow * R; t += kConsumers) {
          float s = 0.f;
          for (int j = 0; j < grp.size; ++j) s += sm.vpart(li & 1, j)[t];
          if (MODE == kFused) {
            vfull[t] = s * sk;
          } else if ((t / R) % grp.size == grp.m && w.ok()) {
            p.v_out[static_cast<size_t>(d[2 + t / R]) * R + (t % R)] = s;
          }
        }
        named_bar(1, kConsumers);
        if (last) cluster_arrive_relaxed();  // all bytes for this CTA have landed (arrive #2)
      }
    }

    if (MODE != kShrink) {
      // ------------------------------------------------------- expand over the N slice
      for (int pass = 0; pass < mp.passes; ++pass) {
        const bool lastp = pass == mp.passes - 1;
        const int wdt = lastp ? mp.w_last : mp.w_full;
        const int cb = lastp ? mp.cb_last : mp.cb_full;
        const int stride = b_row_stride(wdt, kEb);
        const int nch = wdt / kVec;  // compile-time divisor
        int lgc = 0;  // log2 of the lanes that share one 16-byte column chunk
        while (lgc < 5 && (nch << (lgc + 1)) <= kConsumers) ++lgc;
        const int cl_n = 1 << lgc;
        const int my_ch = tid >> lgc, cl = tid & (cl_n - 1);
        const bool active = my_ch < nch;
#pragma unroll
        for (int i = 0; i < RB; ++i)
#pragma unroll
          for (int e = 0; e < kVec; ++e) acc[i][e] = 0.f;
        for (int c0 = 0; c0 < R; c0 += cb, rp.next(NST)) {
          const int rows = max(0, min(cb, rk - c0));  // B rows past the rank were not copied
          w.wait<false>(sm.full(rp.s), rp.par);
          if (active) {
            const uint32_t st = sm.stage_u32(rp.s) + my_ch * 16;
            for (int c = cl; c < rows; c += 2 * cl_n) {  // two B rows in flight per thread
              const int c1 = c + cl_n;
              const bool h1 = c1 < rows;
              float b0[kVec], b1[kVec];
              E::lds(st + c * stride, b0);
              if (h1) {
                E::lds(st + c1 * stride, b1);
              } else {
#pragma unroll
                for (int e = 0; e < kVec; ++e) b1[e] = 0.f;
              }
#pragma unroll
              for (int i = 0; i < RB; ++i) {
                const float v0 = __uint_as_float(lds32(vfull_u32 + 4u * (i * R + c0 + c)));
                const float v1 = h1 ? __uint_as_float(lds32(vfull_u32 + 4u * (i * R + c0 + c1))) : 0.f;
#pragma unroll
                for (int e = 0; e < kVec; ++e) acc[i][e] = fmaf(v1, b1[e], fmaf(v0, b0[e], acc[i][e]));
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.empty(rp.s));
        }
        for (int o = 1; o < cl_n; o <<= 1)
#pragma unroll
          for (int i = 0; i < RB; ++i)
#pragma unroll
            for (int e = 0; e < kVec; ++e) acc[i][e] += __shfl_xor_sync(0xffffffffu, acc[i][e], o);
        // The pass's y rows: add, round once into the y stage, then bulk-store the rows (async
        // proxy: the release arrives that follow do not wait for these global writes).
        w.wait<false>(sm.full(rp.s), rp.par);
        const uint32_t ys = sm.stage_u32(rp.s);
        if (active && cl == 0) {
          const int col = my_ch * kVec;
#pragma unroll
          for (int i = 0; i < RB; ++i) {
            if (i < nrow) {
              float yo[kVec];
              E::lds(ys + (i * wdt + col) * kEb, yo);
#pragma unroll
              for (int e = 0; e < kVec; ++e) yo[e] += acc[i][e];
              E::sts(ys + (i * wdt + col) * kEb, yo);
            }
          }
        }
        fence_proxy_async();  // generic-proxy writes above, read by the bulk store below
        named_bar(1, kConsumers);
        if (tid == 0) {
          if (w.ok()) {
            for (int i = 0; i < nrow; ++i)
              bulk_s2g(static_cast<T*>(p.y) + static_cast<size_t>(d[2 + i]) * p.ldy + mp.n0 +
                           pass * mp.w_full,
                       ys + static_cast<uint32_t>(i * wdt * kEb), static_cast<uint32_t>(wdt * kEb));
            bulk_commit();
          }
          bulk_wait_read();  // the stage may be refilled once the stores have read it
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty(rp.s));
        rp.next(NST);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.fixed(kDescFree0 + (li & 1)));
  }

  __device__ __forceinline__ static void consumer(const Params& p, const Smem& sm,
                                                  const Waiter& w, const Group& grp,
                                                  const MemberPlan& mp, int n_my, int* ctl) {
    RingPos rp;
    rp.init();
    for (int li = 0; li < n_my; ++li) {
      w.wait<false>(sm.fixed(kDescFull0 + (li & 1)), (li >> 1) & 1);
      const int* d = sm.desc(li & 1);
      const int nrow = min(max(d[1], 0), kRowsMax);
      const bool last = li == n_my - 1;
      if (p.adapter_rank) {
        if (nrow <= 1)
          consume_item<1, true>(p, sm, w, grp, mp, li, last, rp, d, nrow, ctl);
        else if (nrow <= 2)
          consume_item<2, true>(p, sm, w, grp, mp, li, last, rp, d, nrow, ctl);
        else
          consume_item<kRowsMax, true>(p, sm, w, grp, mp, li, last, rp, d, nrow, ctl);
      } else {
        if (nrow <= 1)
          consume_item<1, false>(p, sm, w, grp, mp, li, last, rp, d, nrow, ctl);
        else if (nrow <= 2)
          consume_item<2, false>(p, sm, w, grp, mp, li, last, rp, d, nrow, ctl);
        else
          consume_item<kRowsMax, false>(p, sm, w, grp, mp, li, last, rp, d, nrow, ctl);
      }
    }
    // keep every thread's cluster barrier sequence: wait #1, arrive #2 (done per item above
    // when the group exchanges partial products)
    if (MODE != kExpand && !(grp.size > 1 && n_my > 0)) {
      cluster_wait();
      cluster_arrive_relaxed();
    }
  }

  static constexpr bool kTensorRole = sizeof(T) == 2 && R >= 16;

  // Number of CTAs (a multiple of the cluster size) that take the tensor role: all of them
  // when every group is long, else a share proportional to the estimated bytes of each side,
  // leaving at least one cluster to each.  Every CTA computes the same value.
  __device__ __forceinline__ static int tensor_ctas(const Params& p, int S, const int* gcnt,
                                                    int n_items, int n_mt, int N, int* ctl) {
    if (n_mt == 0) return 0;
    if (n_items == 0) return N;
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) {
      ctl[2] = 0;
      ctl[3] = 0;
    }
    __syncthreads();
    int a = 0, b = 0;
    for (int i = tid; i < S; i += NT) {
      const int g = gcnt[i];
      if (g >= p.tc_min_rows) a += g; else b += g;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if (lane == 0) {
      atomicAdd(&ctl[2], a);
      atomicAdd(&ctl[3], b);
    }
    __syncthreads();
    const float act = static_cast<float>(p.h_in + 2 * p.h_out);
    const float wtc = static_cast<float>(ctl[2]) * act;
    const float wcc = static_cast<float>(ctl[3]) * act +
                      static_cast<float>(n_items) * static_cast<float>(p.h_in + p.h_out) * R;
    const int clusters = N / p.C;
    int c_tc = __float2int_rn(static_cast<float>(clusters) * wtc / (wtc + wcc));
    c_tc = max(1, min(c_tc, clusters - 1));
    const long long pairs =  // (m-tile, n-tile) pairs (a shrink has one per m-tile)
        static_cast<long long>(n_mt) * (MODE == kShrink ? 1 : (p.h_out + kTcN - 1) / kTcN);
    if (static_cast<long long>(c_tc) * p.C > pairs)
      c_tc = max(1, static_cast<int>(pairs / p.C));
    return c_tc * p.C;
  }

  __device__ __forceinline__ static void run(const Params& p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    pdl_launch_dependents();  // the next kernel of the stream may start its weight prefetch
    const int tid = threadIdx.x, warp = tid >> 5;
    // Segments to schedule: the table's, or the group count of a plan (its header is checked:
    // every CTA reads the same words, so a bad plan makes the whole grid return here).
    int S = p.S;
    if (p.plan_hdr) {
      const int magic = __ldg(p.plan_hdr), status = __ldg(p.plan_hdr + 1);
      S = __ldg(p.plan_hdr + 3);
      if (magic != kPlanMagic || status != 0 || __ldg(p.plan_hdr + 2) != p.S || S < 0 ||
          S > p.S) {
        if (tid == 0 && blockIdx.x == p.cta0) atomicExch(p.err, kStatusBadPlan);
        return;
      }
    }
    Smem sm;
    sm.init(smem, p);
    int* ctl = reinterpret_cast<int*>(smem + p.off_ctl);
    int* starts = reinterpret_cast<int*>(smem + p.off_tab);
    int* adapters = starts + (p.S + 1);
    int* base = adapters + p.S;
    int* gcnt = base + (p.S + 1);

    if (tid == 0) {  // CUDA-core role barriers (a tensor-role CTA invalidates them again)
      ctl[0] = 0;
      for (int i = kCtlIssued; i <= kCtlPendBar; ++i) ctl[i] = 0;
      for (int s = 0; s < p.nstages; ++s) {
        mbar_init(sm.full(s), 1);
        mbar_init(sm.empty(s), kConsumerWarps);
      }
      mbar_init(sm.fixed(kDescFull0), 1);
      mbar_init(sm.fixed(kDescFull1), 1);
      mbar_init(sm.fixed(kDescFree0), kConsumerWarps);
      mbar_init(sm.fixed(kDescFree1), kConsumerWarps);
      mbar_init(sm.fixed(kNever), 1);
    }
    int* tbase = gcnt + p.S;
    build_schedule<NT>(p, S, starts, adapters, base, gcnt, tbase,
                       reinterpret_cast<int*>(smem + p.off_ring), ctl + 4);
    const int n_items = base[S];
    const int N = p.nctas;                                 // this problem's CTAs...
    const int bx = static_cast<int>(blockIdx.x) - p.cta0;  // ...and this CTA among them
    // Long groups go to the tensor role: the first n_tc CTAs (whole clusters).
    int n_tc = 0;
    if constexpr (kTensorRole) {
      if (p.tc_min_rows < 0x7fffffff) n_tc = tensor_ctas(p, S, gcnt, n_items, tbase[S], N, ctl);
      if (bx < n_tc) {
        if (tid == 0) {  // the barrier words are re-initialised by the tensor role
          for (int s = 0; s < p.nstages; ++s) {
            mbar_inval(sm.full(s));
            mbar_inval(sm.empty(s));
          }
          for (int b : {kDescFull0, kDescFull1, kDescFree0, kDescFree1, kNever})
            mbar_inval(sm.fixed(b));
        }
        fence_proxy_async();  // the ring held the hash table
        // (the tensor role makes its own cluster barriers: one after its barriers are
        // initialised, one before exit)
        TcRole<T, R, MODE, NT>::run(p, S, smem, starts, adapters, gcnt, tbase, ctl, bx, n_tc,
                                    tbase[S]);
        return;
      }
    }
    // A CUDA-core CTA never allocates tensor memory: give up the right at once, so that CTAs
    // of the next kernel can be scheduled beside this one.
    if constexpr (kTensorRole) {
      if (warp == kConsumerWarps) tmem_relinquish();
    }
    const int bid = bx - n_tc;  // index among the CUDA-core CTAs
    const int Nc = N - n_tc;
    // Group size E: each item (one adapter's weights, W bytes) is split over E CTAs so that
    // the busiest CTA finishes first: minimise ceil(n_items E / Nc) x (W / E + X [E > 1]),
    // X (host-set) being the streaming time, in bytes, that the partial-sum exchange through
    // distributed shared memory costs.
    Group grp;
    grp.size = 1;
    {
      const long long W = static_cast<long long>(R) * (p.h_in + p.h_out) * kEb;
      const long long X = p.xchg_bytes;
      long long best = static_cast<long long>((n_items + Nc - 1) / Nc) * W;
      // (E = 2^lg2, so W / E is a shift: a 64-bit division here took ~0.7 us of start-up)
      for (int lg2 = 1; (1 << lg2) <= p.C; ++lg2) {
        const int e = 1 << lg2;
        const long long cost =
            static_cast<long long>((n_items * e + Nc - 1) / Nc) * ((W >> lg2) + X);
        if (cost < best) {
          best = cost;
          grp.size = e;
        }
      }
    }
    const int lg = grp.size == 1 ? 0 : (grp.size == 2 ? 1 : 2);
    grp.m = bid & (grp.size - 1);
    grp.gid = bid >> lg;
    grp.ng = Nc >> lg;
    grp.rank0 = (bx & (p.C - 1)) & ~(grp.size - 1);  // cta0 is a multiple of C
    if (tid == 0) {
      mbar_init(sm.fixed(kVReady0), 1);  // the member's own expect_tx arrival + E partials' bytes
      mbar_init(sm.fixed(kVReady1), 1);
      fence_mbar_init();
    }
    fence_proxy_async();  // the ring held the hash table: order before bulk copies land
    __syncthreads();
    // Cluster barrier protocol (fused / shrink), per thread: arrive #1 here (the barriers that
    // peers write to are initialised; the init fence above publishes them, so the arrival is
    // relaxed) -> wait #1 before the first write to a peer -> arrive #2 (relaxed) once every
    // byte pushed to this CTA has landed -> wait #2 at exit (no CTA leaves while a peer may
    // still write to it).  Peers only ever push (st.async) into this CTA: nothing here is read
    // remotely, so no arrival has to release other writes.
    if (MODE != kExpand) cluster_arrive_relaxed();

    const Waiter w{reinterpret_cast<volatile int*>(ctl), p.err, p.wait_limit_ns};
    if (p.inject_stall) w.wait<false>(sm.fixed(kNever), 0);  // nothing completes it

    const int n_my = (grp.gid < n_items) ? (n_items - grp.gid + grp.ng - 1) / grp.ng : 0;
    const MemberPlan& mp = p.plan[(grp.size - 1) + grp.m];

    if (warp >= kConsumerWarps) {  // the producer, and the warps of the wide geometry that
      if (warp == kConsumerWarps)   // only the tensor role uses
        producer(p, sm, w, grp, mp, starts, adapters, base, gcnt,
                 reinterpret_cast<int4*>(smem + p.off_stab), n_my, ctl, S);
      if (MODE != kExpand) {
        cluster_wait();
        cluster_arrive_relaxed();
      }
    } else {
      consumer(p, sm, w, grp, mp, n_my, ctl);
    }
    __syncthreads();
    if (!w.ok() && tid == 0) {
      // Gave up: before the CTA exits, wait (bounded) for every asynchronous copy into its
      // shared memory -- the last fill of each ring slot, and the partial products that peers
      // of the cluster may still be pushing.  (Bulk stores were waited for as they were issued.)
      const uint32_t issued = static_cast<uint32_t>(ctl[kCtlIssued]);
      const uint32_t par = static_cast<uint32_t>(ctl[kCtlParity]);
      for (int s = 0; s < sm.nst; ++s)
        if ((issued >> s) & 1u) w.drain<false>(sm.full(s), (par >> s) & 1u);
      if (ctl[kCtlPending])
        w.drain<true>(sm.fixed(ctl[kCtlPendBar]), static_cast<uint32_t>(ctl[kCtlPending] - 1));
    }
    __syncthreads();
    if (MODE != kExpand) cluster_wait();
  }
};

// Two CTAs per SM (the default geometry): 288 threads at <= 96 registers.
template <typename T, int R, int MODE>
__global__ void __launch_bounds__(kThreads, 2) sgmv_kernel(const __grid_constant__ Params p) {
  Kernel<T, R, MODE, kThreads>::run(p);
}

// One CTA per SM (SGMV_LONG_BATCH): 416 threads (a second tensor-role epilogue warpgroup).
template <typename T, int R, int MODE>
__global__ void __launch_bounds__(kThreadsWide, 1)
    sgmv_kernel_wide(const __grid_constant__ Params p) {
  Kernel<T, R, MODE, kThreadsWide>::run(p);
}

// Several projections in one launch (lora_apply_multi): problem q runs on CTAs
// [prob[q].cta0, prob[q].cta0 + prob[q].nctas), each with its own weights, activations and
// shared-memory layout, all with the same element type and rank.
struct MultiParams {
  int32_t P;
  Params prob[kMaxProblems];
};

template <typename T, int R>
__global__ void __launch_bounds__(kThreads, 2)
    sgmv_kernel_multi(const __grid_constant__ MultiParams mp) {
  int q = 0;
  while (q + 1 < mp.P && static_cast<int>(blockIdx.x) >= mp.prob[q + 1].cta0) ++q;
  Kernel<T, R, kFused, kThreads>::run(mp.prob[q]);
}

template <typename T, int R>
__global__ void __launch_bounds__(kThreadsWide, 1)
    sgmv_kernel_multi_wide(const __grid_constant__ MultiParams mp) {
  int q = 0;
  while (q + 1 < mp.P && static_cast<int>(blockIdx.x) >= mp.prob[q + 1].cta0) ++q;
  Kernel<T, R, kFused, kThreadsWide>::run(mp.prob[q]);
}

template <typename T, int R>
static const void* multi_kernel_ptr(bool wide) {
  return wide ? reinterpret_cast<const void*>(&sgmv_kernel_multi_wide<T, R>)
              : reinterpret_cast<const void*>(&sgmv_kernel_multi<T, R>);
}

// Host-side handle of one instantiation (for the launch).
template <typename T, int R, int MODE>
static const void* kernel_ptr(bool wide) {
  return wide ? reinterpret_cast<const void*>(&sgmv_kernel_wide<T, R, MODE>)
              : reinterpret_cast<const void*>(&sgmv_kernel<T, R, MODE>);
}

}  // namespace sgmv
