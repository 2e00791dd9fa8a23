// sgmv_pool.cu -- the adapter pool (include/sgmv.h, sgmv_pool_*): a fixed number of device
// slots, each holding one adapter's A and B blocks, filled on demand from host copies.
//
// "Punica Guide: Multi-Tenant LoRA Serving with SGMV", section "Core Innovation 2: Decoupled
// Multi-Tenant Memory Architecture" (dynamic LoRA space allocation: adapter weights are
// streamed from host memory into a GPU pool asynchronously, so that loading a cold adapter
// overlaps the compute of the running batch) and the figure of section "Core Innovation 1"
// (the kernel reaches each adapter through a pointer array).
//
// Design: the caller owns the device slab and the device pointer arrays; the pool owns a
// host-side index (adapter -> slot, least-recently-used order, pins, the last release of each
// slot) and a small ring of pinned staging tables, both made at creation.
// sgmv_pool_acquire makes a batch's adapters resident and pins their slots: misses evict the
// least-recently-used slot that is unpinned and whose last release has completed on the
// device, and enqueue its copies on the copy stream; the compute stream then waits for those
// copies (one event) and the pointer arrays are rewritten on the compute stream, after every
// kernel enqueued before.  sgmv_pool_release unpins the batch's slots and records, on the
// compute stream, when the kernels enqueued so far are done with them.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <list>
#include <mutex>
#include <new>
#include <vector>

#include "sgmv.h"

struct sgmv_pool {
  std::mutex mu;
  int device = 0;
  uint8_t* slab = nullptr;
  int32_t slots = 0, num_adapters = 0;
  size_t a_bytes = 0, b_bytes = 0, slot_bytes = 0;
  std::vector<const void*> host_a, host_b;  // registered host copies, per adapter id
  std::vector<int32_t> slot_of;             // adapter -> slot (-1: not resident)
  std::vector<int32_t> adapter_in;          // slot -> adapter (-1: free)
  std::list<int32_t> lru;                   // slots, least recently used first
  std::vector<std::list<int32_t>::iterator> lru_pos;
  std::vector<cudaEvent_t> done;            // slot -> the last release of a batch reading it
  std::vector<uint8_t> has_done;
  std::vector<int32_t> pins;                // slot -> acquires not yet released
  cudaEvent_t copies = nullptr;             // the last acquire's copies
  static constexpr int kStages = 4;         // pinned host images of A_ptrs then B_ptrs
  uint64_t* stage[kStages] = {};
  cudaEvent_t stage_done[kStages] = {};
  int next_stage = 0;
  uint64_t hits = 0, misses = 0;
};

namespace {

size_t elem_bytes(int dtype) {
  return dtype == SGMV_F32 ? 4 : (dtype == SGMV_F16 || dtype == SGMV_BF16) ? 2 : 0;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// A slot may be refilled once every batch that read it has released it and the kernels before
// that release have completed.
bool slot_idle(sgmv_pool* p, int s) {
  if (p->pins[s] > 0) return false;
  if (!p->has_done[s]) return true;
  const cudaError_t q = cudaEventQuery(p->done[s]);
  if (q == cudaSuccess) return true;
  if (q != cudaErrorNotReady) cudaGetLastError();  // clear a sticky-free error state
  return false;
}

}  // namespace

extern "C" {

size_t sgmv_pool_slot_bytes(int32_t layers, int32_t h_in, int32_t h_out, int32_t r,
                            sgmv_dtype_t dtype) {
  const size_t eb = elem_bytes(dtype);
  if (!eb || layers <= 0 || h_in <= 0 || h_out <= 0 || r <= 0) return 0;
  return up256(static_cast<size_t>(layers) * h_in * r * eb) +
         up256(static_cast<size_t>(layers) * r * h_out * eb);
}

int sgmv_pool_create(sgmv_pool_t** out, void* slab, size_t slab_bytes, int32_t slots,
                     int32_t num_adapters, int32_t layers, int32_t h_in, int32_t h_out,
                     int32_t r, sgmv_dtype_t dtype) {
  if (!out || !slab || slots <= 0 || num_adapters <= 0) return SGMV_EINVAL;
  const size_t sb = sgmv_pool_slot_bytes(layers, h_in, h_out, r, dtype);
  if (!sb) return SGMV_EINVAL;
  if (reinterpret_cast<uintptr_t>(slab) & 255u) return SGMV_EALIGN;
  if (slab_bytes / sb < static_cast<size_t>(slots)) return SGMV_EINVAL;
  sgmv_pool* p = new (std::nothrow) sgmv_pool;
  if (!p) return SGMV_ECUDA;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return SGMV_ECUDA;
  }
  const size_t eb = elem_bytes(dtype);
  p->slab = static_cast<uint8_t*>(slab);
  p->slots = slots;
  p->num_adapters = num_adapters;
  p->a_bytes = static_cast<size_t>(layers) * h_in * r * eb;
  p->b_bytes = static_cast<size_t>(layers) * r * h_out * eb;
  p->slot_bytes = sb;
  p->host_a.assign(num_adapters, nullptr);
  p->host_b.assign(num_adapters, nullptr);
  p->slot_of.assign(num_adapters, -1);
  p->adapter_in.assign(slots, -1);
  p->lru_pos.resize(slots);
  p->done.assign(slots, nullptr);
  p->has_done.assign(slots, 0);
  p->pins.assign(slots, 0);
  for (int s = 0; s < slots; ++s) p->lru_pos[s] = p->lru.insert(p->lru.end(), s);
  bool ok = cudaEventCreateWithFlags(&p->copies, cudaEventDisableTiming) == cudaSuccess;
  for (int s = 0; ok && s < slots; ++s)
    ok = cudaEventCreateWithFlags(&p->done[s], cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < sgmv_pool::kStages; ++i)
    ok = cudaMallocHost(reinterpret_cast<void**>(&p->stage[i]),
                        16 * static_cast<size_t>(num_adapters)) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->stage_done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    sgmv_pool_destroy(p);
    return SGMV_ECUDA;
  }
  *out = p;
  return SGMV_OK;
}

int sgmv_pool_destroy(sgmv_pool_t* p) {
  if (!p) return SGMV_EINVAL;
  int dev = 0;
  const bool switch_dev = cudaGetDevice(&dev) == cudaSuccess && dev != p->device;
  if (switch_dev) cudaSetDevice(p->device);
  for (cudaEvent_t e : p->done)
    if (e) {
      cudaEventSynchronize(e);
      cudaEventDestroy(e);
    }
  if (p->copies) {
    cudaEventSynchronize(p->copies);
    cudaEventDestroy(p->copies);
  }
  for (int i = 0; i < sgmv_pool::kStages; ++i) {
    if (p->stage_done[i]) {
      cudaEventSynchronize(p->stage_done[i]);
      cudaEventDestroy(p->stage_done[i]);
    }
    if (p->stage[i]) cudaFreeHost(p->stage[i]);
  }
  if (switch_dev) cudaSetDevice(dev);
  delete p;
  return SGMV_OK;
}

int sgmv_pool_register(sgmv_pool_t* p, int32_t adapter, const void* host_A,
                       const void* host_B) {
  if (!p || !host_A || !host_B || adapter < 0 || adapter >= p->num_adapters) return SGMV_EINVAL;
  std::lock_guard<std::mutex> lk(p->mu);
  // An adapter already in a slot holds the old weights: drop the mapping so that the next
  // acquire copies the new ones (not while an unreleased batch reads that slot).
  const int s = p->slot_of[adapter];
  if (s >= 0) {
    if (p->pins[s] > 0) return SGMV_EBUSY;
    p->slot_of[adapter] = -1;
    p->adapter_in[s] = -1;
  }
  p->host_a[adapter] = host_A;
  p->host_b[adapter] = host_B;
  return SGMV_OK;
}

int sgmv_pool_acquire(sgmv_pool_t* p, const int32_t* ids, int32_t n, void* d_A_ptrs,
                      void* d_B_ptrs, sgmv_stream_t copy_stream, sgmv_stream_t compute_stream,
                      int32_t* copied) {
  if (!p || n < 0 || (n > 0 && !ids) || !d_A_ptrs || !d_B_ptrs) return SGMV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(d_A_ptrs) & 7u) ||
      (reinterpret_cast<uintptr_t>(d_B_ptrs) & 7u))
    return SGMV_EALIGN;
  std::lock_guard<std::mutex> lk(p->mu);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(copy_stream);
  cudaStream_t ks = reinterpret_cast<cudaStream_t>(compute_stream);
  // The batch's distinct adapters (negative ids carry no adapter).
  std::vector<int32_t> want;
  std::vector<uint8_t> seen(p->num_adapters, 0);
  for (int i = 0; i < n; ++i) {
    const int k = ids[i];
    if (k < 0) continue;
    if (k >= p->num_adapters || !p->host_a[k]) return SGMV_EINVAL;
    if (!seen[k]) {
      seen[k] = 1;
      want.push_back(k);
    }
  }
  if (static_cast<int>(want.size()) > p->slots) return SGMV_ENOSPACE;
  // Hits move to the back of the LRU order first, so that misses never evict them.
  std::vector<int32_t> miss;
  for (int k : want) {
    const int s = p->slot_of[k];
    if (s >= 0) {
      p->lru.splice(p->lru.end(), p->lru, p->lru_pos[s]);
      ++p->hits;
    } else {
      miss.push_back(k);
    }
  }
  // Victims: least recently used slots that hold none of this batch's adapters and that no
  // unfinished batch reads.  Chosen before any copy is enqueued, so a failure changes nothing.
  std::vector<int32_t> victims;
  const size_t keep_from = want.size() - miss.size();  // the last hits in LRU order are ours
  size_t scanned = 0;
  const size_t candidates = p->lru.size() - keep_from;
  for (auto it = p->lru.begin(); victims.size() < miss.size() && scanned < candidates;
       ++it, ++scanned) {
    const int s = *it;
    const int a = p->adapter_in[s];
    if (a >= 0 && seen[a]) continue;
    if (slot_idle(p, s)) victims.push_back(s);
  }
  if (victims.size() < miss.size()) return SGMV_ENOSPACE;
  int rc = SGMV_OK;
  for (size_t j = 0; j < miss.size() && rc == SGMV_OK; ++j) {
    const int k = miss[j], s = victims[j];
    uint8_t* dst = p->slab + static_cast<size_t>(s) * p->slot_bytes;
    if (cudaMemcpyAsync(dst, p->host_a[k], p->a_bytes, cudaMemcpyHostToDevice, cs) !=
            cudaSuccess ||
        cudaMemcpyAsync(dst + up256(p->a_bytes), p->host_b[k], p->b_bytes,
                        cudaMemcpyHostToDevice, cs) != cudaSuccess) {
      rc = SGMV_ECUDA;
      break;
    }
    const int old = p->adapter_in[s];
    if (old >= 0) p->slot_of[old] = -1;
    p->adapter_in[s] = k;
    p->slot_of[k] = s;
    p->lru.splice(p->lru.end(), p->lru, p->lru_pos[s]);
    ++p->misses;
  }
  if (rc != SGMV_OK) return rc;
  for (int k : want) ++p->pins[p->slot_of[k]];  // until sgmv_pool_release
  if (copied) *copied = static_cast<int32_t>(miss.size());
  // The compute stream waits for the copies, then the pointer arrays are rewritten in stream
  // order (after every kernel already enqueued on it has read the previous ones).
  if (!miss.empty() && (cudaEventRecord(p->copies, cs) != cudaSuccess ||
                        cudaStreamWaitEvent(ks, p->copies, 0) != cudaSuccess))
    return SGMV_ECUDA;
  // The host image goes through a ring of pinned staging tables; a table is rewritten only
  // once the copy that last read it has completed.
  const int st = p->next_stage;
  p->next_stage = (st + 1) % sgmv_pool::kStages;
  if (cudaEventSynchronize(p->stage_done[st]) != cudaSuccess) return SGMV_ECUDA;
  uint64_t* tab = p->stage[st];
  const size_t na = static_cast<size_t>(p->num_adapters);
  for (size_t k = 0; k < na; ++k) {
    const int s = p->slot_of[k];
    const uint64_t a =
        s < 0 ? 0 : reinterpret_cast<uint64_t>(p->slab + static_cast<size_t>(s) * p->slot_bytes);
    tab[k] = a;
    tab[na + k] = s < 0 ? 0 : a + up256(p->a_bytes);
  }
  if (cudaMemcpyAsync(d_A_ptrs, tab, na * 8, cudaMemcpyHostToDevice, ks) != cudaSuccess ||
      cudaMemcpyAsync(d_B_ptrs, tab + na, na * 8, cudaMemcpyHostToDevice, ks) != cudaSuccess ||
      cudaEventRecord(p->stage_done[st], ks) != cudaSuccess)
    return SGMV_ECUDA;
  return SGMV_OK;
}

int sgmv_pool_release(sgmv_pool_t* p, const int32_t* ids, int32_t n,
                      sgmv_stream_t compute_stream) {
  if (!p || n < 0 || (n > 0 && !ids)) return SGMV_EINVAL;
  std::lock_guard<std::mutex> lk(p->mu);
  cudaStream_t ks = reinterpret_cast<cudaStream_t>(compute_stream);
  std::vector<uint8_t> seen(p->num_adapters, 0);
  for (int i = 0; i < n; ++i) {
    const int k = ids[i];
    if (k < 0 || k >= p->num_adapters || seen[k]) continue;
    seen[k] = 1;
    const int s = p->slot_of[k];
    if (s < 0 || p->pins[s] == 0) continue;  // not acquired
    if (cudaEventRecord(p->done[s], ks) != cudaSuccess) return SGMV_ECUDA;
    p->has_done[s] = 1;
    --p->pins[s];
  }
  return SGMV_OK;
}

int sgmv_pool_stats(const sgmv_pool_t* p, uint64_t* hits, uint64_t* misses, int32_t* resident) {
  if (!p) return SGMV_EINVAL;
  if (hits) *hits = p->hits;
  if (misses) *misses = p->misses;
  if (resident) {
    int32_t n = 0;
    for (int a : p->adapter_in) n += a >= 0;
    *resident = n;
  }
  return SGMV_OK;
}

}  // extern "C"
