// sgmv_plan.cu -- sgmv_plan / sgmv_plan_size (include/sgmv.h): the adapter grouping of a
// segment table, built once on the device and reused by every planned call of the batch.
//
// "Punica Guide: Multi-Tenant LoRA Serving with SGMV", section "Hardware-Level Optimizations
// in SGMV" (segment descriptors pre-sorted so that each adapter's weights stream once) and
// section "Mathematical Modeling: Throughput Scaling and Kernel Launch Bounds", part 2 (all
// adapter work of a layer in a fixed number of launches, for every layer): the grouping of the
// table does not depend on the layer or on the projection, so it is computed here once per
// batch instead of in every CTA of every call.
//
// Plan layout (int32 words; S = the table's capacity num_segments, max_rows = row capacity):
//   [0] magic   [1] status (0 ok, 1 more than max_rows rows)   [2] S   [3] G groups
//   [4] rows listed   [5] max_rows   [6..15] zero
//   [16, 16 + S + 1)            group row offsets g_starts[0..G]
//   [17 + S, 17 + 2 S)          group adapters g_adapter[0..G)
//   [17 + 2 S, 17 + 2 S + max_rows)  row list: the token indices of group 0, then group 1, ...
// Groups are the distinct adapter ids >= 0 of non-empty segments, in the order of their first
// segment; a group's rows are its segments' rows, segment after segment.  The compute kernels
// read this table as a segment table with one segment per group (sgmv_core.cuh).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sgmv.h"
#include "sgmv_core.cuh"

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanWarps = kPlanThreads / 32;

int hash_slots_for(int S) {
  int hs = 64;  // power of two, load factor <= 2/3
  while (hs < S + S / 2 + 2) hs <<= 1;
  return hs;
}

size_t plan_smem_bytes(int S, int HS) {
  // starts[S+1], adapters[S], slot[S], segoff[S], hkey/hoff[HS], hlead[HS], hcnt/hrun[HS],
  // scan partials
  return 4 * (static_cast<size_t>(4 * S + 1) + 3 * static_cast<size_t>(HS) + 2 * kPlanWarps + 4);
}

__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const int32_t* __restrict__ ss, const int32_t* __restrict__ sa, int S, int HS,
                int max_rows, int32_t* __restrict__ plan) {
  extern __shared__ int sm[];
  int* starts = sm;
  int* adapters = starts + S + 1;
  int* slot = adapters + S;
  int* segoff = slot + S;
  int* hkey = segoff + S;  // key, then (after grouping) the group's first row in the list
  int* hlead = hkey + HS;
  int* hcnt = hlead + HS;  // rows per group, then the running row count of the listing
  int* wpart = hcnt + HS;  // [kPlanWarps][2] scan partials, then totals
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* g_starts = plan + sgmv::kPlanHeader;
  int32_t* g_adapter = g_starts + S + 1;
  int32_t* rows = g_adapter + S;

  for (int i = tid; i <= S; i += kPlanThreads) {
    starts[i] = ss[i];
    if (i < S) adapters[i] = sa[i];
  }
  for (int h = tid; h < HS; h += kPlanThreads) {
    hkey[h] = -1;
    hlead[h] = 0x7fffffff;
    hcnt[h] = 0;
  }
  __syncthreads();
  // 1. Hash every non-empty segment with an adapter by its id: the lead (first segment) and
  //    the row count of each adapter's group.
  for (int i = tid; i < S; i += kPlanThreads) {
    const int k = adapters[i];
    const int len = starts[i + 1] - starts[i];
    int h = -1;
    if (k >= 0 && len > 0) {
      h = static_cast<int>((static_cast<uint32_t>(k) * 0x9E3779B1u >> 12) &
                           static_cast<uint32_t>(HS - 1));
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
  // 2. Number the groups in the order of their leads and give each its first row in the list:
  //    an exclusive scan over the segments of (is lead, rows of the group if lead).
  const int per = (S + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(tid * per, S), hi = min(lo + per, S);
  int cg = 0, cr = 0;
  for (int i = lo; i < hi; ++i) {
    const int h = slot[i];
    if (h >= 0 && hlead[h] == i) {
      ++cg;
      cr += hcnt[h];
    }
  }
  int ig = cg, ir = cr;  // inclusive warp scan
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ig, o), b = __shfl_up_sync(0xffffffffu, ir, o);
    if (lane >= o) {
      ig += a;
      ir += b;
    }
  }
  if (lane == 31) {
    wpart[2 * warp] = ig;
    wpart[2 * warp + 1] = ir;
  }
  __syncthreads();
  if (tid == 0) {
    int g = 0, r = 0;
    for (int w = 0; w < kPlanWarps; ++w) {
      const int a = wpart[2 * w], b = wpart[2 * w + 1];
      wpart[2 * w] = g;
      wpart[2 * w + 1] = r;
      g += a;
      r += b;
    }
    wpart[2 * kPlanWarps] = g;
    wpart[2 * kPlanWarps + 1] = r;
  }
  __syncthreads();
  const int G = wpart[2 * kPlanWarps], n_rows = wpart[2 * kPlanWarps + 1];
  if (n_rows > max_rows) {  // the caller's capacity is too small: an invalid plan
    if (tid == 0) {
      plan[0] = sgmv::kPlanMagic;
      plan[1] = 1;
      plan[2] = S;
      plan[3] = 0;
      plan[4] = n_rows;
      plan[5] = max_rows;
      for (int i = 6; i < sgmv::kPlanHeader; ++i) plan[i] = 0;
    }
    return;
  }
  int g = wpart[2 * warp] + ig - cg, r = wpart[2 * warp + 1] + ir - cr;
  for (int i = lo; i < hi; ++i) {
    const int h = slot[i];
    if (h >= 0 && hlead[h] == i) {
      g_starts[g] = r;
      g_adapter[g] = adapters[i];
      hkey[h] = r;  // the group's first row in the list
      ++g;
      r += hcnt[h];
    }
  }
  __syncthreads();
  for (int h = tid; h < HS; h += kPlanThreads) hcnt[h] = 0;  // now the running row count
  __syncthreads();
  // 3. Each segment's row offset inside its group, in segment order: one warp walks the table
  //    32 segments at a time; lanes of the same group add up the lengths of the lower lanes.
  if (warp == 0) {
    for (int b = 0; b < S; b += 32) {
      const int i = b + lane;
      const int h = i < S ? slot[i] : -1;
      const int len = h >= 0 ? starts[i + 1] - starts[i] : 0;
      const unsigned same = __match_any_sync(0xffffffffu, h);
      int pre = 0;
      for (int j = 0; j < 32; ++j) {
        const int lj = __shfl_sync(0xffffffffu, len, j);
        if (j < lane && ((same >> j) & 1u)) pre += lj;
      }
      const int off = h >= 0 ? hcnt[h] + pre : 0;
      __syncwarp();
      if (h >= 0 && (same >> lane) == 1u) hcnt[h] = off + len;  // highest lane of its group
      if (i < S) segoff[i] = off;
      __syncwarp();
    }
  }
  __syncthreads();
  // 4. The row list: every row of every grouped segment, at its group's first row + the
  //    segment's offset in the group.
  for (int i = warp; i < S; i += kPlanWarps) {
    const int h = slot[i];
    if (h < 0) continue;
    const int len = starts[i + 1] - starts[i];
    const int dst = hkey[h] + segoff[i];
    for (int q = lane; q < len; q += 32) rows[dst + q] = starts[i] + q;
  }
  if (tid == 0) {
    g_starts[G] = n_rows;
    plan[0] = sgmv::kPlanMagic;
    plan[1] = 0;
    plan[2] = S;
    plan[3] = G;
    plan[4] = n_rows;
    plan[5] = max_rows;
    for (int i = 6; i < sgmv::kPlanHeader; ++i) plan[i] = 0;
  }
}

// ---- lora_apply_static_plan: the plan in a fixed device array instead of caller memory ----
// Some callers cannot allocate device memory when they call the library (see the header): the
// plan, the only scratch memory of the planned path, then lives in this file-scope array,
// sized for SGMV_MAX_SEGMENTS segments and SGMV_STATIC_PLAN_MAX_ROWS rows.  Every device that
// loads the library holds it until the process exits.  The plan kernel rewrites every word the
// apply kernel reads, so nothing in it has to be cleared between calls.
constexpr size_t kStaticPlanWords = static_cast<size_t>(sgmv::kPlanHeader) +
                                    2 * static_cast<size_t>(SGMV_MAX_SEGMENTS) + 1 +
                                    static_cast<size_t>(SGMV_STATIC_PLAN_MAX_ROWS);
static __device__ __align__(256) int32_t g_static_plan[kStaticPlanWords];

constexpr int kMaxDevices = 64;
std::once_flag g_static_once[kMaxDevices];
int32_t* g_static_addr[kMaxDevices] = {};
int g_static_rc[kMaxDevices] = {};

// The array's device address on the current device, looked up once per device (with that
// device current).  In host code the array's name is only a host-side stand-in.
int static_plan_address(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SGMV_ECUDA;
  std::call_once(g_static_once[dev], [dev] {
    void* ptr = nullptr;
    const cudaError_t rc = cudaGetSymbolAddress(&ptr, g_static_plan);
    g_static_rc[dev] = rc == cudaSuccess && ptr ? SGMV_OK : SGMV_ECUDA;
    g_static_addr[dev] = static_cast<int32_t*>(ptr);
  });
  if (g_static_rc[dev] != SGMV_OK) return g_static_rc[dev];
  *out = g_static_addr[dev];
  return SGMV_OK;
}

}  // namespace

extern "C" {

int lora_apply_static_plan(void* y, int32_t ldy, const void* x, int32_t ldx,
                           const void* const* A_ptrs, const void* const* B_ptrs,
                           const int32_t* seg_starts, const int32_t* seg_adapter,
                           int32_t num_segments, int32_t max_rows, int32_t layer_idx,
                           int32_t h_in, int32_t h_out, int32_t r, float scale,
                           sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream) {
  if (num_segments < 0 || max_rows < 0 || !seg_starts || (num_segments > 0 && !seg_adapter))
    return SGMV_EINVAL;
  if (num_segments > SGMV_MAX_SEGMENTS || max_rows > SGMV_STATIC_PLAN_MAX_ROWS)
    return SGMV_EUNSUPPORTED;
  // The apply kernel reads the plan that the kernel just before it writes: it must wait for
  // that kernel, so it cannot be launched as its programmatic dependent.
  if (flags & SGMV_OVERLAP_PRIOR) return SGMV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(seg_starts) & 3u) ||
      (reinterpret_cast<uintptr_t>(seg_adapter) & 3u))
    return SGMV_EALIGN;
  // Every argument of the apply call is checked before anything is enqueued: with no segments
  // the planned call runs its host checks only and never reads the plan pointer (any non-null
  // 16-byte-aligned value passes its own check).
  const void* const kChecksOnly = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  int rc = lora_apply_planned(y, ldy, x, ldx, A_ptrs, B_ptrs, kChecksOnly, 0, layer_idx, h_in,
                              h_out, r, scale, dtype, flags, stream);
  if (rc != SGMV_OK) return rc;
  if (num_segments == 0) return SGMV_OK;
  int32_t* plan = nullptr;
  if ((rc = static_plan_address(&plan)) != SGMV_OK) return rc;
  if ((rc = sgmv_plan(seg_starts, seg_adapter, num_segments, max_rows, plan,
                      sizeof(int32_t) * kStaticPlanWords, stream)) != SGMV_OK)
    return rc;
  return lora_apply_planned(y, ldy, x, ldx, A_ptrs, B_ptrs, plan, num_segments, layer_idx, h_in,
                            h_out, r, scale, dtype, flags, stream);
}

size_t sgmv_plan_size(int32_t num_segments, int32_t max_rows) {
  if (num_segments < 0 || max_rows < 0 || num_segments > SGMV_MAX_SEGMENTS) return 0;
  return 4 * (static_cast<size_t>(sgmv::kPlanHeader) + 2 * static_cast<size_t>(num_segments) +
              1 + static_cast<size_t>(max_rows));
}

int sgmv_plan(const int32_t* seg_starts, const int32_t* seg_adapter, int32_t num_segments,
              int32_t max_rows, void* plan, size_t plan_bytes, sgmv_stream_t stream) {
  if (num_segments < 0 || max_rows < 0 || !seg_starts || !plan ||
      (num_segments > 0 && !seg_adapter))
    return SGMV_EINVAL;
  if (num_segments > SGMV_MAX_SEGMENTS) return SGMV_EUNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(plan) & 15u) ||
      (reinterpret_cast<uintptr_t>(seg_starts) & 3u) ||
      (reinterpret_cast<uintptr_t>(seg_adapter) & 3u))
    return SGMV_EALIGN;
  if (plan_bytes < sgmv_plan_size(num_segments, max_rows)) return SGMV_EINVAL;
  const int HS = hash_slots_for(num_segments);
  const size_t smem = plan_smem_bytes(num_segments, HS);
  // (the attribute is per device; setting it is a host-side call, and a plan is built once
  // per batch)
  if (cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return SGMV_ECUDA;
  plan_kernel<<<1, kPlanThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
      seg_starts, seg_adapter, num_segments, HS, max_rows, static_cast<int32_t*>(plan));
  return cudaGetLastError() == cudaSuccess ? SGMV_OK : SGMV_ECUDA;
}

}  // extern "C"
