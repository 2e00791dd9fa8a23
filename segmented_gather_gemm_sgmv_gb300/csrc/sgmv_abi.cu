// sgmv_abi.cu -- the C ABI declared in include/sgmv.h: argument checks, launch geometry,
// kernel attributes, the table-validation kernel and the library's device error word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "sgmv.h"
#include "sgmv_core.cuh"
#include "sgmv_launch.h"

namespace {

// Written by kernels whose bounded wait ran out (SGMV_ETIMEOUT); read by sgmv_get_error.
__device__ int g_sgmv_error = 0;

constexpr int kMaxDevices = 64;
constexpr size_t kPairSmem = 114688;  // 112 KB: two CTAs fit on an SM (228 KB), so the next
                                      // kernel of the stream can start beside this one
constexpr size_t kMaxSmem = 232448;   // 227 KB: large segment tables (one CTA per SM)
constexpr int kWideMaxSegments = 64;  // long-batch tables up to this size use the wide kernel
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

struct KernelCache {  // per kernel instantiation
  const void* fn = nullptr;
  size_t smem_set = 0;
  int cluster = 0;     // the grid size below was computed for this cluster size...
  size_t smem_q = 0;   // ...and this shared-memory size
  int max_clusters = 0;
};

struct DeviceState {
  std::once_flag once;
  int init_rc = SGMV_ECUDA;  // written once, under `once`
  int sms = 0;
  int* err = nullptr;
  std::atomic<uint64_t> wait_ns{kDefaultWaitNs};
  std::atomic<int> inject{0};
  // dtype, mode (fused, shrink, expand, multi-projection fused), rank index, geometry
  // (SGMV_LONG_BATCH); guarded by g_mu
  KernelCache cache[3][4][4][2];
};

std::mutex g_mu;  // guards the kernel caches
DeviceState g_dev[kMaxDevices];

constexpr int kMaxStages = 16;

// Launch-geometry and routing constants (chosen by measurement on GB300; fixed at build time).
// Adapter groups of at least half a 128-row tile may use the tensor cores (measured: 64 beats
// 128 on the 70B mix, 16 and 32 tie) ...
constexpr int kTcMinRows = 64;
// ... when their CUDA-core items would re-read at least this many MB of weights (ceil(rows / 4)
// items x the adapter's A and B bytes).
constexpr int kTcMinMB = 32;
// The shrink-only launch streams A alone, half the bytes of a fused item at the same rank: it
// takes the tensor cores from a lower volume (measured on the prefill mix, rank 64, groups of
// 142-195 rows: on the CUDA cores those groups made sgmv_shrink 60 us; rank-16 decode groups
// of up to 256 rows (8 MB) stay faster on the CUDA cores).
constexpr int kTcMinMBShrink = 16;
// Cost of one partial-sum exchange through distributed shared memory, in streamed KB (the
// group-size rule of the CUDA-core role).
constexpr int kXchgKB = 64;

// Ring stage size.  Rank 16: 20 KB, i.e. an A chunk of 512 rows plus its x columns for four
// rows, with five stages in the ring (24 KB stages hold the same 512-row chunks, four at a
// time: measured 5.8 vs 6.4 us per chained decode call).  Larger ranks: 24 KB (measured on the
// 70B mix, rank 64: 136 vs 138 us).
int stage_kb_for(int r) { return r <= 16 ? 20 : 24; }

int rank_index(int r) {
  switch (r) {
    case 8: return 0;
    case 16: return 1;
    case 32: return 2;
    case 64: return 3;
    default: return -1;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled, looked up once through the runtime (no link against the driver).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Tensor map of a row-major [rows][cols] 16-bit matrix: boxes of 64 columns x box_rows rows
// with the 128-byte swizzle (8-row atoms of 1024 bytes).  The row extent is not known to the library
// (the call carries no M); the kernel only addresses rows named by the segment table, so the
// map declares the largest row count TMA accepts.  Columns past `cols` read as zero.
bool encode_rows(sgmv::TmaMap* out, const void* base, int cols, int ld, int dtype, int box_rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  CUtensorMap m;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), 0x7fffffffull};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};  // row stride, bytes
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult rc = fn(&m, dtype == SGMV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (rc != CUDA_SUCCESS) return false;
  static_assert(sizeof(m) == sizeof(*out), "tensor map size");
  std::memcpy(out, &m, sizeof(m));
  return true;
}
size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Per-device state of the current device, set up once (thread-safe) on first use.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SGMV_ECUDA;
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&st, dev] {
    void* p = nullptr;
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        cudaGetSymbolAddress(&p, g_sgmv_error) == cudaSuccess) {
      st.err = static_cast<int*>(p);
      st.init_rc = SGMV_OK;
    }
  });
  if (st.init_rc != SGMV_OK) return st.init_rc;
  *out = &st;
  return SGMV_OK;
}

const void* kernel_for(int dtype, int mode, int r, bool wide) {
  switch (dtype) {
    case SGMV_F32: return sgmv::kernel_f32(mode, r, wide);
    case SGMV_F16: return sgmv::kernel_f16(mode, r, wide);
    case SGMV_BF16: return sgmv::kernel_bf16(mode, r, wide);
    default: return nullptr;
  }
}

const void* multi_kernel_for(int dtype, int r, bool wide) {
  switch (dtype) {
    case SGMV_F32: return sgmv::kernel_multi_f32(r, wide);
    case SGMV_F16: return sgmv::kernel_multi_f16(r, wide);
    case SGMV_BF16: return sgmv::kernel_multi_bf16(r, wide);
    default: return nullptr;
  }
}

struct Problem {
  int mode;
  int dtype;
  int r;
  int S;
  int layer;
  int h_in;
  int h_out;
  float scale;
};

void slice(int n, int parts, int m, int* lo, int* hi) {
  const int units = n / 8;  // slices start on multiples of 8 elements (16-byte aligned)
  *lo = units * m / parts * 8;
  *hi = units * (m + 1) / parts * 8;
}

// B rows per chunk of an expand pass of width w: as many as a stage holds, balanced.
int pass_rows(int r, int stage_bytes, int w, int eb) {
  const int cap = std::min(r, stage_bytes / (w * eb + 16));
  const int n = (r + cap - 1) / cap;
  return (r + n - 1) / n;
}

// Chunk plan of member m of a group of E CTAs (the kernel indexes these, so it does no
// division by runtime values).
sgmv::MemberPlan member_plan(const Problem& pb, int E, int m, int kb, int wmax, int stage_bytes,
                             int eb) {
  sgmv::MemberPlan mp = {};
  int k1 = 0, n1 = 0;
  slice(pb.h_in, E, m, &mp.k0, &k1);
  slice(pb.h_out, E, m, &mp.n0, &n1);
  mp.kc = pb.mode == sgmv::kExpand ? 0 : k1 - mp.k0;
  mp.nc = pb.mode == sgmv::kShrink ? 0 : n1 - mp.n0;
  mp.nA = (mp.kc + kb - 1) / kb;
  mp.kbe = mp.nA > 0 ? ((mp.kc + mp.nA - 1) / mp.nA + 7) / 8 * 8 : kb;
  mp.nA = (mp.kc + mp.kbe - 1) / mp.kbe;
  mp.passes = (mp.nc + wmax - 1) / wmax;
  mp.total = mp.nA + (pb.mode == sgmv::kExpand ? 1 : 0);
  if (mp.passes > 0) {
    mp.w_full = wmax;
    mp.cb_full = pass_rows(pb.r, stage_bytes, wmax, eb);
    mp.nb_full = (pb.r + mp.cb_full - 1) / mp.cb_full;
    mp.w_last = mp.nc - (mp.passes - 1) * wmax;
    mp.cb_last = pass_rows(pb.r, stage_bytes, mp.w_last, eb);
    mp.nb_last = (pb.r + mp.cb_last - 1) / mp.cb_last;
    mp.total += (mp.passes - 1) * (mp.nb_full + 1) + mp.nb_last + 1;
  }
  return mp;
}

// Lays out shared memory and fills the geometry part of the kernel parameters.  The launch
// cluster is kMaxGroup CTAs; the kernel itself picks how many of them share an item.
int plan_geometry(const Problem& pb, size_t budget, sgmv::Params& p, size_t* smem_out) {
  const int eb = pb.dtype == SGMV_F32 ? 4 : 2;
  const int vec = 16 / eb;
  const int C = sgmv::kMaxGroup;
  const int rmax = sgmv::kRowsMax;
  const int stage_bytes = stage_kb_for(pb.r) * 1024;
  // A rows per stage, followed by the same rows' columns of up to rmax x rows.
  const int kb = (stage_bytes / ((pb.r + rmax) * eb)) / 8 * 8;
  // Expand pass width: one thread per 16 bytes of a B row, and rmax y rows must fit a stage.
  const int wmax = std::min(sgmv::kConsumers * vec, stage_bytes / (rmax * eb)) / 8 * 8;
  if (kb < 8 || wmax < 8 || stage_bytes < wmax * eb + 16 || stage_bytes < rmax * pb.r * 4)
    return SGMV_EUNSUPPORTED;
  int hs = 64;  // hash slots: power of two, load factor <= 2/3
  while (hs < pb.S + pb.S / 2 + 2) hs <<= 1;

  size_t off = 0;
  p.off_bars = static_cast<uint32_t>(off);
  off += up(8 * (2 * kMaxStages + sgmv::kNumFixedBars), 16);
  p.off_ctl = static_cast<uint32_t>(off);
  off += 128;
  p.desc_ints = static_cast<int32_t>(up(2 + rmax, 4));
  p.off_desc = static_cast<uint32_t>(off);
  off += 2 * 4 * p.desc_ints;
  // starts[S+1], adapters[S], base[S+1], gcnt[S], tbase[S+1]
  p.off_tab = static_cast<uint32_t>(off);
  off += up(4 * (5 * static_cast<size_t>(pb.S) + 3), 16);
  p.off_vpart = static_cast<uint32_t>(off);  // [2][kMaxGroup][rmax][r] fp32 partials
  off += 2 * sgmv::kMaxGroup * 4 * rmax * pb.r;
  p.off_vfull = static_cast<uint32_t>(off);
  off += 4 * rmax * pb.r;
  p.off_red = static_cast<uint32_t>(off);
  off += 4 * sgmv::kConsumerWarps * rmax * pb.r;
  // producer's stage-descriptor table (16 bytes per stage of the longest member plan)
  int max_total = 0;
  for (int E = 1, slot = 0; E <= C; E <<= 1)
    for (int m = 0; m < E; ++m, ++slot) {
      p.plan[slot] = member_plan(pb, E, m, kb, wmax, stage_bytes, eb);
      max_total = std::max(max_total, p.plan[slot].total);
    }
  p.off_stab = static_cast<uint32_t>(up(off, 16));
  off = p.off_stab + 16 * static_cast<size_t>(max_total);
  p.off_ring = static_cast<uint32_t>(up(off, 1024));
  // As many ring stages as the budget holds (the ring also hosts the transient hash table).
  const size_t scratch = 4 * (static_cast<size_t>(pb.S) + 3 * hs);
  if (p.off_ring + std::max<size_t>(scratch, 2 * static_cast<size_t>(stage_bytes)) > budget)
    return SGMV_EUNSUPPORTED;
  int nst = static_cast<int>((budget - p.off_ring) / stage_bytes);
  nst = std::min(std::max(nst, 2), kMaxStages);
  const size_t ring = std::max<size_t>(static_cast<size_t>(nst) * stage_bytes, scratch);
  off = p.off_ring + ring;
  if (off > budget) return SGMV_EUNSUPPORTED;

  p.C = C;
  p.xchg_bytes = kXchgKB * 1024;
  p.nstages = nst;
  p.stage_bytes = stage_bytes;
  p.kb = kb;
  p.hash_slots = hs;
  *smem_out = off;
  return SGMV_OK;
}

// ---- launch set-up, shared by the single, planned and multi-projection entry points ----

bool tensor_capable(const Problem& pb, uint32_t flags) {
  return pb.dtype != SGMV_F32 && pb.r >= 16 && !(flags & SGMV_NO_TENSOR_CORES);
}

// Shared-memory layout and the per-problem kernel parameters that do not depend on the grid.
// Returns the bytes of dynamic shared memory this problem needs in this geometry.
int setup_problem(const DeviceState* st, const Problem& pb, sgmv::Params& p, uint32_t flags,
                  size_t* smem_out) {
  const size_t budget = (flags & SGMV_LONG_BATCH) ? kMaxSmem : kPairSmem;
  size_t smem = 0;
  int rc = plan_geometry(pb, budget, p, &smem);
  if (rc == SGMV_EUNSUPPORTED) rc = plan_geometry(pb, kMaxSmem, p, &smem);
  if (rc != SGMV_OK) return rc;
  p.err = st->err;
  p.S = pb.S;
  p.layer = pb.layer;
  p.h_in = pb.h_in;
  p.h_out = pb.h_out;
  p.scale = pb.scale;
  p.wait_limit_ns = st->wait_ns.load(std::memory_order_relaxed);
  p.inject_stall = st->inject.load(std::memory_order_relaxed);
  p.dependent = (flags & SGMV_OVERLAP_PRIOR) ? 1 : 0;
  // Tensor role (16-bit types, r >= 16; every mode): it uses none of the CUDA-core scratch
  // areas, so its row table sits at off_vpart and its ring of 24 KB slots right after it, up to
  // the end of the budget (the launch then always takes the whole budget).
  p.tc_base = static_cast<uint32_t>(
      up(p.off_vpart + (2 * sgmv::kTcRows + 4) * sizeof(int), 1024));
  if (tensor_capable(pb, flags) && smem <= budget) smem = budget;
  *smem_out = smem;
  return SGMV_OK;
}

// Clusters of C CTAs that fit at once for this kernel and shared-memory size (one CTA per SM
// per kernel), cached per instantiation.  Also sets the kernel's attributes.
int grid_for(DeviceState* st, KernelCache& kc, const void* fn, int threads, size_t smem,
             bool clustered, int C, int* grid, bool dense = false) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (kc.smem_set < smem) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return SGMV_ECUDA;
    if (clustered && C > 8 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess)
      return SGMV_ECUDA;
    kc.smem_set = smem;
  }
  if (kc.cluster != C || kc.smem_q != smem) {
    int n = 0;
    if (clustered) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      cfg.gridDim = dim3(static_cast<unsigned>(C * st->sms), 1, 1);
      cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
      cfg.dynamicSmemBytes = smem;
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(C);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) return SGMV_ECUDA;
    } else {
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) !=
          cudaSuccess)
        return SGMV_ECUDA;
      n = per_sm * st->sms / C;
    }
    n = std::min(n, std::max(1, st->sms / C));  // one CTA per SM per kernel
    if (n <= 0) return SGMV_EUNSUPPORTED;
    kc.cluster = C;
    kc.smem_q = smem;
    kc.max_clusters = n;
  }
  *grid = kc.max_clusters * C;
  // SGMV_DENSE_GRID: two CTAs of the call per SM.  Two default-geometry CTAs fit on an SM (that
  // is what lets the next kernel of the stream start beside this one); the occupancy query
  // answers one cluster slot per SM for this size, so the count is set directly.  No CTA waits
  // on a CTA of another cluster, so a grid that did not fit would only run in two waves.
  if (dense && smem <= kPairSmem) *grid = std::max(*grid, 2 * (st->sms / C) * C);
  return SGMV_OK;
}

// The grid-dependent part of a problem's parameters: its CTA range and the tensor role (ring
// slots, tensor maps, routing threshold), which needs at least two clusters and three slots.
int finish_problem(const Problem& pb, sgmv::Params& p, uint32_t flags, size_t smem, int cta0,
                   int nctas, bool wide_kernel) {
  p.cta0 = cta0;
  p.nctas = nctas;
  p.tc_min_rows = 0x7fffffff;
  p.tc_slots = 0;
  const size_t xchg = pb.mode != sgmv::kExpand ? sgmv::kTcXchgBytes : 0;  // split-K buffers
  if (tensor_capable(pb, flags) && nctas >= 2 * p.C && smem > p.tc_base + xchg) {
    int slots = std::min<int>(static_cast<int>((smem - p.tc_base - xchg) / sgmv::kTcSlot),
                              (2 * kMaxStages + sgmv::kNumFixedBars - sgmv::kTcNumFixed) / 2);
    // Two epilogue groups take alternate n-tiles: with an even slot count the previous use of
    // every slot within an m-tile belongs to the same group, so no group can wait on a slot
    // whose previous fill (another group's) has not landed yet (parity waits see one phase).
    if (wide_kernel) slots &= ~1;
    p.tc_xchg = p.tc_base + static_cast<uint32_t>(slots) * sgmv::kTcSlot;
    if (slots >= 3) {
      const bool need_x = pb.mode != sgmv::kExpand, need_y = pb.mode != sgmv::kShrink;
      if ((need_x && (!encode_rows(&p.tmap_x128, p.x, pb.h_in, p.ldx, pb.dtype, 128) ||
                      !encode_rows(&p.tmap_x8, p.x, pb.h_in, p.ldx, pb.dtype, 8) ||
                      !encode_rows(&p.tmap_x64, p.x, pb.h_in, p.ldx, pb.dtype, 64) ||
                      !encode_rows(&p.tmap_x32, p.x, pb.h_in, p.ldx, pb.dtype, 32) ||
                      !encode_rows(&p.tmap_x16, p.x, pb.h_in, p.ldx, pb.dtype, 16))) ||
          (need_y && (!encode_rows(&p.tmap_y128, p.y, pb.h_out, p.ldy, pb.dtype, 128) ||
                      !encode_rows(&p.tmap_y8, p.y, pb.h_out, p.ldy, pb.dtype, 8) ||
                      !encode_rows(&p.tmap_y64, p.y, pb.h_out, p.ldy, pb.dtype, 64) ||
                      !encode_rows(&p.tmap_y32, p.y, pb.h_out, p.ldy, pb.dtype, 32) ||
                      !encode_rows(&p.tmap_y16, p.y, pb.h_out, p.ldy, pb.dtype, 16))))
        return SGMV_ECUDA;
      // The CUDA-core path streams a group's weights once per item of 4 rows (mostly from
      // L2); the tensor path streams them once per 128-row tile (split over the cluster).
      // Measured on GB300: small-rank decode groups (256 rows, r = 16, h = 4096: 17 MB of
      // weight re-reads) run faster on the CUDA cores; prefill groups (r = 64, >= 60 MB) and
      // the hot groups of the 70B mix (r = 64, h = 8192) faster on the tensor cores.
      const double w = static_cast<double>(pb.r) * 2.0 *
                       ((pb.mode != sgmv::kExpand ? pb.h_in : 0) +
                        (pb.mode != sgmv::kShrink ? pb.h_out : 0));
      const double min_mb = pb.mode == sgmv::kShrink ? kTcMinMBShrink : kTcMinMB;
      const double items = std::ceil(min_mb * 1048576.0 / w);
      p.tc_min_rows = (flags & SGMV_TENSOR_CORES_ALWAYS)
                          ? 64
                          : static_cast<int>(std::min(
                                1e9, std::max<double>(kTcMinRows, 4.0 * items)));
      p.tc_slots = slots;
    }
  }
  return SGMV_OK;
}

int launch_kernel(const void* fn, int grid, int threads, size_t smem, bool clustered, int C,
                  uint32_t flags, void* arg, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  unsigned na = 0;
  if (clustered) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(C);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (flags & SGMV_OVERLAP_PRIOR) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  void* args[] = {arg};
  return cudaLaunchKernelExC(&cfg, fn, args) == cudaSuccess ? SGMV_OK : SGMV_ECUDA;
}

// The 416-thread kernel (a second tensor-role epilogue warpgroup) measured faster where the
// tensor role dominates (prefill_mixed, 8 segments: 61.1 -> 58.3 us) and slower on the
// CUDA-core role (the 70B mix, 482 segments: 101.0 -> 105.6 us); a table of many segments
// means many decode rows, so those keep the 288-thread kernel.
bool use_wide_kernel(const Problem& pb, uint32_t flags) {
  return (flags & SGMV_LONG_BATCH) && pb.S <= kWideMaxSegments;
}

// One problem, one launch.
int launch(const Problem& pb, sgmv::Params& p, uint32_t flags, cudaStream_t stream) {
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != SGMV_OK) return rc;
  size_t smem = 0;
  if ((rc = setup_problem(st, pb, p, flags, &smem)) != SGMV_OK) return rc;
  const bool wide_kernel = use_wide_kernel(pb, flags);
  const void* fn = kernel_for(pb.dtype, pb.mode, pb.r, wide_kernel);
  const int threads = wide_kernel ? sgmv::kThreadsWide : sgmv::kThreads;
  if (!fn) return SGMV_EUNSUPPORTED;
  const bool clustered = pb.mode != sgmv::kExpand;
  int grid = 0;
  rc = grid_for(st, st->cache[pb.dtype][pb.mode][rank_index(pb.r)][wide_kernel ? 1 : 0], fn,
                threads, smem, clustered, p.C, &grid, (flags & SGMV_DENSE_GRID) != 0);
  if (rc != SGMV_OK) return rc;
  if ((rc = finish_problem(pb, p, flags, smem, 0, grid, wide_kernel)) != SGMV_OK) return rc;
  return launch_kernel(fn, grid, threads, smem, clustered, p.C, flags, &p, stream);
}

bool flags_ok(uint32_t flags) {
  if (flags & ~static_cast<uint32_t>(SGMV_OVERLAP_PRIOR | SGMV_NO_TENSOR_CORES |
                                     SGMV_TENSOR_CORES_ALWAYS | SGMV_LONG_BATCH |
                                     SGMV_DENSE_GRID))
    return false;
  return !((flags & SGMV_NO_TENSOR_CORES) && (flags & SGMV_TENSOR_CORES_ALWAYS));
}

int check_common(int num_segments, const void* seg_starts, const void* seg_adapter,
                 int layer_idx, int r, int dtype) {
  if (num_segments < 0 || layer_idx < 0) return SGMV_EINVAL;
  if (dtype != SGMV_F32 && dtype != SGMV_F16 && dtype != SGMV_BF16) return SGMV_EINVAL;
  if (!seg_starts || (num_segments > 0 && !seg_adapter)) return SGMV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(seg_starts) & 3u) ||
      (reinterpret_cast<uintptr_t>(seg_adapter) & 3u))
    return SGMV_EALIGN;
  if (rank_index(r) < 0) return SGMV_EUNSUPPORTED;
  if (num_segments > SGMV_MAX_SEGMENTS) return SGMV_EUNSUPPORTED;
  return SGMV_OK;
}

int check_hidden(int h) {
  if (h <= 0) return SGMV_EINVAL;
  if (h > SGMV_MAX_HIDDEN) return SGMV_EUNSUPPORTED;
  if (h % 8) return SGMV_EALIGN;
  return SGMV_OK;
}

// Row stride (elements) of x or y: at least the row length, a multiple of 8 elements (rows
// start 16-byte aligned for the bulk and tensor copies), at most SGMV_MAX_LD.
int check_ld(int ld, int h) {
  if (ld < h) return SGMV_EINVAL;
  if (ld > SGMV_MAX_LD) return SGMV_EUNSUPPORTED;
  if (ld % 8) return SGMV_EALIGN;
  return SGMV_OK;
}

// Checks table entries on the device; see sgmv_validate in include/sgmv.h.
__global__ void validate_kernel(const int32_t* ss, const int32_t* sa, int S, int num_adapters,
                                int M, int32_t* err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  int bits = 0;
  if (i == 0) {
    if (ss[0] < 0) bits |= 2;
    if (ss[S] > M) bits |= 4;
  }
  if (i < S) {
    if (ss[i + 1] < ss[i]) bits |= 1;
    if (sa[i] >= num_adapters) bits |= 8;
  }
  if (bits) atomicOr(err, bits);
}

// Checks the weight pointers of every adapter a non-empty segment uses; see
// sgmv_validate_pointers in include/sgmv.h.  Reads pointer values only, never what they point to.
__global__ void validate_ptrs_kernel(const void* const* A_ptrs, const void* const* B_ptrs,
                                     const int32_t* ss, const int32_t* sa, int S,
                                     int num_adapters, int32_t* err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= S) return;
  const int k = sa[i];
  if (k < 0 || k >= num_adapters || ss[i + 1] <= ss[i]) return;
  int bits = 0;
  if (A_ptrs) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(A_ptrs[k]);
    if (a == 0 || (a & 15u)) bits |= 16;
  }
  if (B_ptrs) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(B_ptrs[k]);
    if (b == 0 || (b & 15u)) bits |= 32;
  }
  if (bits) atomicOr(err, bits);
}

}  // namespace

namespace sgmv {
int device_context(int** err, int* sms, uint64_t* wait_ns, int* inject_stall) {
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != SGMV_OK) return rc;
  *err = st->err;
  *sms = st->sms;
  *wait_ns = st->wait_ns.load(std::memory_order_relaxed);
  *inject_stall = st->inject.load(std::memory_order_relaxed);
  return SGMV_OK;
}
}  // namespace sgmv

extern "C" {

int lora_apply(void* y, const void* x, const void* const* A_ptrs, const void* const* B_ptrs,
               const int32_t* seg_starts, const int32_t* seg_adapter, int32_t num_segments,
               int32_t layer_idx, int32_t h_in, int32_t h_out, int32_t r, float scale,
               sgmv_dtype_t dtype, sgmv_stream_t stream) {
  return lora_apply_ex(y, x, A_ptrs, B_ptrs, seg_starts, seg_adapter, num_segments, layer_idx,
                       h_in, h_out, r, scale, dtype, 0u, stream);
}

int lora_apply_ex(void* y, const void* x, const void* const* A_ptrs, const void* const* B_ptrs,
                  const int32_t* seg_starts, const int32_t* seg_adapter, int32_t num_segments,
                  int32_t layer_idx, int32_t h_in, int32_t h_out, int32_t r, float scale,
                  sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream) {
  return lora_apply_strided(y, h_out, x, h_in, A_ptrs, B_ptrs, seg_starts, seg_adapter,
                            num_segments, layer_idx, h_in, h_out, r, scale, dtype, flags, stream);
}

int lora_apply_strided(void* y, int32_t ldy, const void* x, int32_t ldx,
                       const void* const* A_ptrs, const void* const* B_ptrs,
                       const int32_t* seg_starts, const int32_t* seg_adapter,
                       int32_t num_segments, int32_t layer_idx, int32_t h_in, int32_t h_out,
                       int32_t r, float scale, sgmv_dtype_t dtype, uint32_t flags,
                       sgmv_stream_t stream) {
  if (!flags_ok(flags)) return SGMV_EINVAL;
  int rc = check_common(num_segments, seg_starts, seg_adapter, layer_idx, r, dtype);
  if (rc != SGMV_OK) return rc;
  if (!y || !x || !A_ptrs || !B_ptrs) return SGMV_EINVAL;
  if ((rc = check_hidden(h_in)) != SGMV_OK || (rc = check_hidden(h_out)) != SGMV_OK) return rc;
  if ((rc = check_ld(ldx, h_in)) != SGMV_OK || (rc = check_ld(ldy, h_out)) != SGMV_OK) return rc;
  if (!aligned16(y) || !aligned16(x) || (reinterpret_cast<uintptr_t>(A_ptrs) & 7u) ||
      (reinterpret_cast<uintptr_t>(B_ptrs) & 7u))
    return SGMV_EALIGN;
  if (num_segments == 0) return SGMV_OK;
  sgmv::Params p = {};
  p.y = y;
  p.x = x;
  p.ldx = ldx;
  p.ldy = ldy;
  p.A_ptrs = A_ptrs;
  p.B_ptrs = B_ptrs;
  p.seg_starts = seg_starts;
  p.seg_adapter = seg_adapter;
  const Problem pb{sgmv::kFused, dtype, r, num_segments, layer_idx, h_in, h_out, scale};
  return launch(pb, p, flags, reinterpret_cast<cudaStream_t>(stream));
}

int sgmv_shrink(float* v, const void* x, const void* const* A_ptrs, const int32_t* seg_starts,
                const int32_t* seg_adapter, int32_t num_segments, int32_t layer_idx,
                int32_t h_in, int32_t r, sgmv_dtype_t dtype, sgmv_stream_t stream) {
  return sgmv_shrink_ex(v, x, A_ptrs, seg_starts, seg_adapter, num_segments, layer_idx, h_in, r,
                        dtype, 0u, stream);
}

int sgmv_shrink_ex(float* v, const void* x, const void* const* A_ptrs,
                   const int32_t* seg_starts, const int32_t* seg_adapter, int32_t num_segments,
                   int32_t layer_idx, int32_t h_in, int32_t r, sgmv_dtype_t dtype,
                   uint32_t flags, sgmv_stream_t stream) {
  return sgmv_shrink_strided(v, x, h_in, A_ptrs, seg_starts, seg_adapter, num_segments,
                             layer_idx, h_in, r, dtype, flags, stream);
}

int sgmv_shrink_strided(float* v, const void* x, int32_t ldx, const void* const* A_ptrs,
                        const int32_t* seg_starts, const int32_t* seg_adapter,
                        int32_t num_segments, int32_t layer_idx, int32_t h_in, int32_t r,
                        sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream) {
  if (!flags_ok(flags)) return SGMV_EINVAL;
  int rc = check_common(num_segments, seg_starts, seg_adapter, layer_idx, r, dtype);
  if (rc != SGMV_OK) return rc;
  if (!v || !x || !A_ptrs) return SGMV_EINVAL;
  if ((rc = check_hidden(h_in)) != SGMV_OK) return rc;
  if ((rc = check_ld(ldx, h_in)) != SGMV_OK) return rc;
  if (!aligned16(v) || !aligned16(x) || (reinterpret_cast<uintptr_t>(A_ptrs) & 7u))
    return SGMV_EALIGN;
  if (num_segments == 0) return SGMV_OK;
  sgmv::Params p = {};
  p.x = x;
  p.ldx = ldx;
  p.ldy = 8;
  p.v_out = v;
  p.A_ptrs = A_ptrs;
  p.seg_starts = seg_starts;
  p.seg_adapter = seg_adapter;
  const Problem pb{sgmv::kShrink, dtype, r, num_segments, layer_idx, h_in, 8, 1.0f};
  return launch(pb, p, flags, reinterpret_cast<cudaStream_t>(stream));
}

int sgmv_expand(void* y, const float* v, const void* const* B_ptrs, const int32_t* seg_starts,
                const int32_t* seg_adapter, int32_t num_segments, int32_t layer_idx, int32_t r,
                int32_t h_out, float scale, sgmv_dtype_t dtype, sgmv_stream_t stream) {
  return sgmv_expand_ex(y, v, B_ptrs, seg_starts, seg_adapter, num_segments, layer_idx, r, h_out,
                        scale, dtype, 0u, stream);
}

int sgmv_expand_ex(void* y, const float* v, const void* const* B_ptrs,
                   const int32_t* seg_starts, const int32_t* seg_adapter, int32_t num_segments,
                   int32_t layer_idx, int32_t r, int32_t h_out, float scale, sgmv_dtype_t dtype,
                   uint32_t flags, sgmv_stream_t stream) {
  return sgmv_expand_strided(y, h_out, v, B_ptrs, seg_starts, seg_adapter, num_segments,
                             layer_idx, r, h_out, scale, dtype, flags, stream);
}

int sgmv_expand_strided(void* y, int32_t ldy, const float* v, const void* const* B_ptrs,
                        const int32_t* seg_starts, const int32_t* seg_adapter,
                        int32_t num_segments, int32_t layer_idx, int32_t r, int32_t h_out,
                        float scale, sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream) {
  if (!flags_ok(flags)) return SGMV_EINVAL;
  int rc = check_common(num_segments, seg_starts, seg_adapter, layer_idx, r, dtype);
  if (rc != SGMV_OK) return rc;
  if (!y || !v || !B_ptrs) return SGMV_EINVAL;
  if ((rc = check_hidden(h_out)) != SGMV_OK) return rc;
  if ((rc = check_ld(ldy, h_out)) != SGMV_OK) return rc;
  if (!aligned16(y) || !aligned16(v) || (reinterpret_cast<uintptr_t>(B_ptrs) & 7u))
    return SGMV_EALIGN;
  if (num_segments == 0) return SGMV_OK;
  sgmv::Params p = {};
  p.y = y;
  p.ldx = 8;
  p.ldy = ldy;
  p.v_in = v;
  p.B_ptrs = B_ptrs;
  p.seg_starts = seg_starts;
  p.seg_adapter = seg_adapter;
  const Problem pb{sgmv::kExpand, dtype, r, num_segments, layer_idx, 8, h_out, scale};
  return launch(pb, p, flags, reinterpret_cast<cudaStream_t>(stream));
}

// ---- planned calls (a plan from sgmv_plan instead of the segment table) ----------------

namespace {
int check_plan_args(const void* plan, int32_t num_segments) {
  if (!plan || num_segments < 0) return SGMV_EINVAL;
  if (num_segments > SGMV_MAX_SEGMENTS) return SGMV_EUNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(plan) & 15u) return SGMV_EALIGN;
  return SGMV_OK;
}

// Points the kernel at the plan's group table (one segment per adapter group) and row list.
void use_plan(sgmv::Params& p, const void* plan, int32_t S) {
  const int32_t* h = static_cast<const int32_t*>(plan);
  p.plan_hdr = h;
  p.seg_starts = h + sgmv::kPlanHeader;
  p.seg_adapter = h + sgmv::kPlanHeader + S + 1;
  p.rowmap = h + sgmv::kPlanHeader + 2 * S + 1;
}
}  // namespace

int lora_apply_planned(void* y, int32_t ldy, const void* x, int32_t ldx,
                       const void* const* A_ptrs, const void* const* B_ptrs, const void* plan,
                       int32_t num_segments, int32_t layer_idx, int32_t h_in, int32_t h_out,
                       int32_t r, float scale, sgmv_dtype_t dtype, uint32_t flags,
                       sgmv_stream_t stream) {
  if (!flags_ok(flags)) return SGMV_EINVAL;
  int rc = check_plan_args(plan, num_segments);
  if (rc != SGMV_OK) return rc;
  if ((rc = check_common(num_segments, plan, plan, layer_idx, r, dtype)) != SGMV_OK) return rc;
  if (!y || !x || !A_ptrs || !B_ptrs) return SGMV_EINVAL;
  if ((rc = check_hidden(h_in)) != SGMV_OK || (rc = check_hidden(h_out)) != SGMV_OK) return rc;
  if ((rc = check_ld(ldx, h_in)) != SGMV_OK || (rc = check_ld(ldy, h_out)) != SGMV_OK) return rc;
  if (!aligned16(y) || !aligned16(x) || (reinterpret_cast<uintptr_t>(A_ptrs) & 7u) ||
      (reinterpret_cast<uintptr_t>(B_ptrs) & 7u))
    return SGMV_EALIGN;
  if (num_segments == 0) return SGMV_OK;
  sgmv::Params p = {};
  p.y = y;
  p.x = x;
  p.ldx = ldx;
  p.ldy = ldy;
  p.A_ptrs = A_ptrs;
  p.B_ptrs = B_ptrs;
  use_plan(p, plan, num_segments);
  const Problem pb{sgmv::kFused, dtype, r, num_segments, layer_idx, h_in, h_out, scale};
  return launch(pb, p, flags, reinterpret_cast<cudaStream_t>(stream));
}

int sgmv_shrink_planned(float* v, const void* x, int32_t ldx, const void* const* A_ptrs,
                        const void* plan, int32_t num_segments, int32_t layer_idx, int32_t h_in,
                        int32_t r, sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream) {
  if (!flags_ok(flags)) return SGMV_EINVAL;
  int rc = check_plan_args(plan, num_segments);
  if (rc != SGMV_OK) return rc;
  if ((rc = check_common(num_segments, plan, plan, layer_idx, r, dtype)) != SGMV_OK) return rc;
  if (!v || !x || !A_ptrs) return SGMV_EINVAL;
  if ((rc = check_hidden(h_in)) != SGMV_OK) return rc;
  if ((rc = check_ld(ldx, h_in)) != SGMV_OK) return rc;
  if (!aligned16(v) || !aligned16(x) || (reinterpret_cast<uintptr_t>(A_ptrs) & 7u))
    return SGMV_EALIGN;
  if (num_segments == 0) return SGMV_OK;
  sgmv::Params p = {};
  p.x = x;
  p.ldx = ldx;
  p.ldy = 8;
  p.v_out = v;
  p.A_ptrs = A_ptrs;
  use_plan(p, plan, num_segments);
  const Problem pb{sgmv::kShrink, dtype, r, num_segments, layer_idx, h_in, 8, 1.0f};
  return launch(pb, p, flags, reinterpret_cast<cudaStream_t>(stream));
}

int sgmv_expand_planned(void* y, int32_t ldy, const float* v, const void* const* B_ptrs,
                        const void* plan, int32_t num_segments, int32_t layer_idx, int32_t r,
                        int32_t h_out, float scale, sgmv_dtype_t dtype, uint32_t flags,
                        sgmv_stream_t stream) {
  if (!flags_ok(flags)) return SGMV_EINVAL;
  int rc = check_plan_args(plan, num_segments);
  if (rc != SGMV_OK) return rc;
  if ((rc = check_common(num_segments, plan, plan, layer_idx, r, dtype)) != SGMV_OK) return rc;
  if (!y || !v || !B_ptrs) return SGMV_EINVAL;
  if ((rc = check_hidden(h_out)) != SGMV_OK) return rc;
  if ((rc = check_ld(ldy, h_out)) != SGMV_OK) return rc;
  if (!aligned16(y) || !aligned16(v) || (reinterpret_cast<uintptr_t>(B_ptrs) & 7u))
    return SGMV_EALIGN;
  if (num_segments == 0) return SGMV_OK;
  sgmv::Params p = {};
  p.y = y;
  p.ldx = 8;
  p.ldy = ldy;
  p.v_in = v;
  p.B_ptrs = B_ptrs;
  use_plan(p, plan, num_segments);
  const Problem pb{sgmv::kExpand, dtype, r, num_segments, layer_idx, 8, h_out, scale};
  return launch(pb, p, flags, reinterpret_cast<cudaStream_t>(stream));
}

int lora_apply_multi(const sgmv_projection_t* proj, int32_t num_proj, const void* plan,
                     int32_t num_segments, int32_t layer_idx, int32_t r, sgmv_dtype_t dtype,
                     uint32_t flags, sgmv_stream_t stream) {
  if (!flags_ok(flags) || !proj || num_proj < 1) return SGMV_EINVAL;
  if (num_proj > SGMV_MAX_PROJECTIONS) return SGMV_EUNSUPPORTED;
  int rc = check_plan_args(plan, num_segments);
  if (rc != SGMV_OK) return rc;
  if ((rc = check_common(num_segments, plan, plan, layer_idx, r, dtype)) != SGMV_OK) return rc;
  for (int q = 0; q < num_proj; ++q) {
    const sgmv_projection_t& j = proj[q];
    if (!j.y || !j.x || !j.A_ptrs || !j.B_ptrs) return SGMV_EINVAL;
    if ((rc = check_hidden(j.h_in)) != SGMV_OK || (rc = check_hidden(j.h_out)) != SGMV_OK)
      return rc;
    if ((rc = check_ld(j.ldx, j.h_in)) != SGMV_OK || (rc = check_ld(j.ldy, j.h_out)) != SGMV_OK)
      return rc;
    if (!aligned16(j.y) || !aligned16(j.x) || (reinterpret_cast<uintptr_t>(j.A_ptrs) & 7u) ||
        (reinterpret_cast<uintptr_t>(j.B_ptrs) & 7u))
      return SGMV_EALIGN;
  }
  if (num_segments == 0) return SGMV_OK;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != SGMV_OK) return rc;
  static_assert(sgmv::kMaxProblems == SGMV_MAX_PROJECTIONS, "projection limit");
  sgmv::MultiParams mp;
  std::memset(&mp, 0, sizeof(mp));
  mp.P = num_proj;
  Problem pbs[sgmv::kMaxProblems];
  size_t smem = 0;
  for (int q = 0; q < num_proj; ++q) {
    const sgmv_projection_t& j = proj[q];
    sgmv::Params& p = mp.prob[q];
    p.y = j.y;
    p.x = j.x;
    p.ldx = j.ldx;
    p.ldy = j.ldy;
    p.A_ptrs = j.A_ptrs;
    p.B_ptrs = j.B_ptrs;
    use_plan(p, plan, num_segments);
    pbs[q] = Problem{sgmv::kFused, dtype, r, num_segments, layer_idx, j.h_in, j.h_out, j.scale};
    size_t sq = 0;
    if ((rc = setup_problem(st, pbs[q], p, flags, &sq)) != SGMV_OK) return rc;
    smem = std::max(smem, sq);
  }
  const bool wide_kernel = use_wide_kernel(pbs[0], flags);
  const void* fn = multi_kernel_for(dtype, r, wide_kernel);
  if (!fn) return SGMV_EUNSUPPORTED;
  const int threads = wide_kernel ? sgmv::kThreadsWide : sgmv::kThreads;
  const int C = mp.prob[0].C;
  int grid = 0;
  rc = grid_for(st, st->cache[dtype][3][rank_index(r)][wide_kernel ? 1 : 0], fn, threads, smem,
                true, C, &grid, (flags & SGMV_DENSE_GRID) != 0);
  if (rc != SGMV_OK) return rc;
  // Clusters per projection, in proportion to an estimate of its bytes: the weights of an
  // adapter ((h_in + h_out) r) plus the activations of its rows (h_in + 2 h_out per row; ~4 rows
  // per adapter, ~128 for SGMV_LONG_BATCH launches), at least one cluster each.
  const int clusters = grid / C;
  if (clusters < num_proj) return SGMV_EUNSUPPORTED;
  const double rows = (flags & SGMV_LONG_BATCH) ? 128.0 : 4.0;
  double cost[sgmv::kMaxProblems], total = 0.0;
  for (int q = 0; q < num_proj; ++q) {
    cost[q] = static_cast<double>(pbs[q].h_in + pbs[q].h_out) * r +
              rows * (pbs[q].h_in + 2.0 * pbs[q].h_out);
    total += cost[q];
  }
  int share[sgmv::kMaxProblems], given = 0;
  for (int q = 0; q < num_proj; ++q) {
    share[q] = std::max(1, static_cast<int>((clusters - num_proj) * cost[q] / total) + 1);
    given += share[q];
  }
  for (int q = 0; given > clusters; q = (q + 1) % num_proj)  // trim (never below one)
    if (share[q] > 1) {
      --share[q];
      --given;
    }
  for (int q = 0; given < clusters; q = (q + 1) % num_proj) {  // hand out the remainder
    ++share[q];
    ++given;
  }
  int cta0 = 0;
  for (int q = 0; q < num_proj; ++q) {
    if ((rc = finish_problem(pbs[q], mp.prob[q], flags, smem, cta0, share[q] * C,
                             wide_kernel)) != SGMV_OK)
      return rc;
    cta0 += share[q] * C;
  }
  return launch_kernel(fn, grid, threads, smem, true, C, flags, &mp,
                       reinterpret_cast<cudaStream_t>(stream));
}

int lora_apply_ranked(void* y, int32_t ldy, const void* x, int32_t ldx,
                      const void* const* A_ptrs, const void* const* B_ptrs,
                      const int32_t* adapter_rank, const float* adapter_scale,
                      const int32_t* seg_starts, const int32_t* seg_adapter, const void* plan,
                      int32_t num_segments, int32_t layer_idx, int32_t h_in, int32_t h_out,
                      int32_t r_max, sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream) {
  if (!flags_ok(flags)) return SGMV_EINVAL;
  if (!adapter_rank || !adapter_scale) return SGMV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(adapter_rank) & 3u) ||
      (reinterpret_cast<uintptr_t>(adapter_scale) & 3u))
    return SGMV_EALIGN;
  int rc = SGMV_OK;
  if (plan) {
    if ((rc = check_plan_args(plan, num_segments)) != SGMV_OK) return rc;
    rc = check_common(num_segments, plan, plan, layer_idx, r_max, dtype);
  } else {
    rc = check_common(num_segments, seg_starts, seg_adapter, layer_idx, r_max, dtype);
  }
  if (rc != SGMV_OK) return rc;
  if (!y || !x || !A_ptrs || !B_ptrs) return SGMV_EINVAL;
  if ((rc = check_hidden(h_in)) != SGMV_OK || (rc = check_hidden(h_out)) != SGMV_OK) return rc;
  if ((rc = check_ld(ldx, h_in)) != SGMV_OK || (rc = check_ld(ldy, h_out)) != SGMV_OK) return rc;
  if (!aligned16(y) || !aligned16(x) || (reinterpret_cast<uintptr_t>(A_ptrs) & 7u) ||
      (reinterpret_cast<uintptr_t>(B_ptrs) & 7u))
    return SGMV_EALIGN;
  if (num_segments == 0) return SGMV_OK;
  sgmv::Params p = {};
  p.y = y;
  p.x = x;
  p.ldx = ldx;
  p.ldy = ldy;
  p.A_ptrs = A_ptrs;
  p.B_ptrs = B_ptrs;
  p.adapter_rank = adapter_rank;
  p.adapter_scale = adapter_scale;
  if (plan) {
    use_plan(p, plan, num_segments);
  } else {
    p.seg_starts = seg_starts;
    p.seg_adapter = seg_adapter;
  }
  const Problem pb{sgmv::kFused, dtype, r_max, num_segments, layer_idx, h_in, h_out, 1.0f};
  return launch(pb, p, flags, reinterpret_cast<cudaStream_t>(stream));
}

int sgmv_validate(const int32_t* seg_starts, const int32_t* seg_adapter, int32_t num_segments,
                  int32_t num_adapters, int32_t M, int32_t* d_err, sgmv_stream_t stream) {
  if (num_segments < 0 || !seg_starts || !d_err || (num_segments > 0 && !seg_adapter))
    return SGMV_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(d_err, 0, sizeof(int32_t), s) != cudaSuccess) return SGMV_ECUDA;
  const int threads = 256;
  const int blocks = std::max(1, (num_segments + threads - 1) / threads);
  validate_kernel<<<blocks, threads, 0, s>>>(seg_starts, seg_adapter, num_segments, num_adapters,
                                             M, d_err);
  return cudaGetLastError() == cudaSuccess ? SGMV_OK : SGMV_ECUDA;
}

int sgmv_validate_pointers(const void* const* A_ptrs, const void* const* B_ptrs,
                           const int32_t* seg_starts, const int32_t* seg_adapter,
                           int32_t num_segments, int32_t num_adapters, int32_t* d_err,
                           sgmv_stream_t stream) {
  if (num_segments < 0 || num_adapters < 0 || !seg_starts || !d_err ||
      (num_segments > 0 && !seg_adapter) || (!A_ptrs && !B_ptrs))
    return SGMV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(A_ptrs) & 7u) || (reinterpret_cast<uintptr_t>(B_ptrs) & 7u))
    return SGMV_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(d_err, 0, sizeof(int32_t), s) != cudaSuccess) return SGMV_ECUDA;
  if (num_segments == 0) return SGMV_OK;
  const int threads = 256;
  const int blocks = (num_segments + threads - 1) / threads;
  validate_ptrs_kernel<<<blocks, threads, 0, s>>>(A_ptrs, B_ptrs, seg_starts, seg_adapter,
                                                  num_segments, num_adapters, d_err);
  return cudaGetLastError() == cudaSuccess ? SGMV_OK : SGMV_ECUDA;
}

int sgmv_get_error(int32_t* host_err, int32_t clear, sgmv_stream_t stream) {
  if (!host_err) return SGMV_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_sgmv_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return SGMV_ECUDA;
  *host_err = v;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_sgmv_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return SGMV_ECUDA;
  }
  return SGMV_OK;
}

int sgmv_set_wait_limit(uint64_t limit_ns, int32_t inject_stall) {
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != SGMV_OK) return rc;
  st->wait_ns.store(limit_ns ? limit_ns : kDefaultWaitNs, std::memory_order_relaxed);
  st->inject.store(inject_stall ? 1 : 0, std::memory_order_relaxed);
  return SGMV_OK;
}

const char* sgmv_status_string(int status) {
  switch (status) {
    case SGMV_OK: return "SGMV_OK";
    case SGMV_EINVAL: return "SGMV_EINVAL: invalid argument";
    case SGMV_EALIGN: return "SGMV_EALIGN: misaligned pointer or size";
    case SGMV_EUNSUPPORTED: return "SGMV_EUNSUPPORTED: rank or size outside the supported range";
    case SGMV_ECUDA: return "SGMV_ECUDA: CUDA runtime error";
    case SGMV_ETIMEOUT: return "SGMV_ETIMEOUT: a device-side wait ran out";
    case SGMV_EPLAN: return "SGMV_EPLAN: a planned call was given an invalid plan";
    case SGMV_ENOSPACE: return "SGMV_ENOSPACE: too few free adapter-pool slots for the batch";
    case SGMV_EBUSY: return "SGMV_EBUSY: the adapter's slot is read by an unreleased batch";
    default: return "unknown status";
  }
}

int sgmv_version(void) { return 200; }

}  // extern "C"
