// sgmv_base.cu -- lora_apply_base: the base projection of every row with the LoRA term of its
// adapter added in the same kernel, so that y is written once instead of read and rewritten.
//
// Operation ("Punica Guide: Multi-Tenant LoRA Serving with SGMV", section "The Heterogeneous
// Batching Bottleneck": y_i = x_i W0 + (alpha/r) x_i A_k B_k, and the figure of that section
// in which the base GEMM hands its output to the fused SGMV kernel; here the two are one
// kernel):
//     y[t] = x[t] . W0^T + scale * v[t] . B_k     for the rows t of segments with adapter k
//     y[t] = x[t] . W0^T                          for every other row t < M
// with W0 stored one row per output feature ([h_out][h_in], a linear layer's weight) and
// v = x . A_k computed just before by the library's shrink (sgmv_shrink_strided) into a
// caller-provided fp32 workspace.
//
// GB300 design: a persistent kernel, one CTA per SM, over output tiles of 128 rows x 256
// columns (tile t: m-tile t mod n_mt, n-tile t div n_mt, so the CTAs in flight share the
// same W0 columns in L2).
//   warp 0     one thread issues TMA loads into a ring of 3 stages {x [128 x 64], W0 [256 x
//              64]}, both K-major with the 128-byte swizzle.
//   warp 1     owns the TMEM allocation (two 256-column fp32 accumulators, so one tile's
//              epilogue overlaps the next tile's main loop); one thread issues
//              tcgen05.mma (M 128, N 256, K 16) over h_in, then the LoRA rounds of the tile:
//              per distinct adapter k of the tile's rows, D += [scale*v]_hi . B_k and
//              D += [scale*v]_lo . B_k (v split into two 16-bit parts, rows of other adapters
//              zero), as four N = 64 MMAs per K step of 16.
//   warps 2-5  the epilogue: they build each LoRA round's operands in shared memory (the
//              16-bit parts of scale * v, K-major; B_k's rows for the tile's 256 columns,
//              MN-major), then read the finished accumulator (tcgen05.ld), round it to the
//              output type and store it.
// Every wait is bounded; a wait that runs out sets the library's error word and the CTA
// winds down (waiting, bounded, for its own copies and MMAs) before freeing TMEM.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <cstring>
#include <type_traits>

#include "sgmv.h"
#include "sgmv_launch.h"
#include "sgmv_ptx.cuh"

namespace sgmv_base {

using namespace sgmv;

constexpr int kBM = 128;               // rows per tile (MMA M, TMEM lanes)
constexpr int kBN = 256;               // output columns per tile (MMA N of the base product)
constexpr int kBK = 64;                // h_in per stage: one 128-byte row of 16-bit values
constexpr int kStages = 3;
constexpr int kXBytes = kBM * kBK * 2;             // 16 KB
constexpr int kWBytes = kBN * kBK * 2;             // 32 KB
constexpr int kStageBytes = kXBytes + kWBytes;     // 48 KB
constexpr int kVPart = kBM * 128;                  // one 16-bit part of scale * v (16 KB)
constexpr int kBBlock = 64 * 128;                  // B_k rows for 64 columns, up to 64 rows
constexpr int kLoraBytes = 2 * kVPart + 4 * kBBlock;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr int kStatusTimeout = -5;  // SGMV_ETIMEOUT

// barrier indices (8 bytes each) after the LoRA area
enum Bar : int { kFull0 = 0, kEmpty0 = kStages, kAccFull0 = 2 * kStages, kAccEmpty0 = kAccFull0 + 2,
                 kLoraFull = kAccEmpty0 + 2, kLoraEmpty, kDrain, kNever, kNumBars };
// control words (ints) after the barriers
enum Ctl : int { kAbort = 0, kTmem, kCmd, kIssued, kParity, kEpiOk0, kEpiOk1, kNumCtl = 8 };
constexpr int kSmemBytes = 1024 /* alignment slack */ + kStages * kStageBytes + kLoraBytes +
                           8 * kNumBars + 4 * kNumCtl;

struct alignas(64) Map {
  uint8_t b[128];
};

struct BaseParams {
  Map tmap_x;  // x [M][h_in], boxes of 64 columns x 128 rows
  Map tmap_w;  // W0 [h_out][h_in], boxes of 64 columns x 256 rows
  void* y;
  const float* v;  // [M][r] fp32 (rows of segments with an adapter)
  const void* const* B_ptrs;
  const int32_t* seg_starts;
  const int32_t* seg_adapter;
  int* err;
  unsigned long long wait_ns;
  int S, M, h_in, h_out, r, layer, ldy;
  int n_mt, n_tiles, k_steps;
  float scale;
  int wait_prior_x;  // wait for the previous kernel before the first x load
  int inject_stall;
};

// Bounded waits on this CTA's barriers (the library's convention: a wait that runs out flags
// the CTA and sets the device error word; after that, waits return false at once).
struct Wait {
  volatile int* abort;
  int* err;
  unsigned long long limit;
  __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity) const {
    if (*abort) return false;
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (true) {
#pragma unroll 1
      for (int i = 0; i < 8; ++i)
        if (mbar_try(bar, parity)) return true;
      if (*abort) return false;
      if (now_ns() - t0 > limit) {
        *abort = 1;
        atomicExch(err, kStatusTimeout);
        return false;
      }
    }
  }
  // after giving up: bounded wait for a phase, ignoring the flag
  __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
    const uint64_t t0 = now_ns();
    while (!mbar_try(bar, parity))
      if (now_ns() - t0 > limit) return false;
    return true;
  }
};

// Byte offset of 16-byte chunk c of row m in a block of 128-byte rows, 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128(int m, int c) {
  return static_cast<uint32_t>((m >> 3) * 1024 + (m & 7) * 128 + ((c ^ (m & 7)) << 4));
}

// Number of offsets ss[0..S] that are <= t (the offsets are non-decreasing).
__device__ __forceinline__ int offsets_at_most(const int32_t* ss, int S, int t) {
  int lo = 0, hi = S + 1;  // answer in [lo, hi]
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(ss + mid) <= t) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Index of the segment that holds row t (-1: none).  Offsets are non-decreasing.
__device__ __forceinline__ int segment_of(const int32_t* ss, int S, int t) {
  if (S <= 0 || t < __ldg(ss) || t >= __ldg(ss + S)) return -1;
  int lo = 0, hi = S;  // ss[lo] <= t < ss[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(ss + mid) <= t) lo = mid; else hi = mid;
  }
  return lo;
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (std::is_same_v<T, __half>) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}
template <typename T>
__device__ __forceinline__ float round_to(float a) {
  if constexpr (std::is_same_v<T, __half>) return __half2float(__float2half_rn(a));
  else return __bfloat162float(__float2bfloat16_rn(a));
}

template <typename T, int RK>
struct Kernel {
  static constexpr bool kBf16 = std::is_same_v<T, __nv_bfloat16>;
  static constexpr uint32_t kIdBase = idesc_f16(kBf16, false, kBM, kBN);
  static constexpr uint32_t kIdDelta = idesc_f16(kBf16, true, kBM, 64);

  struct Smem {
    uint32_t ring, lora, bars;
    int* ctl;
    __device__ __forceinline__ uint32_t x(int s) const { return ring + s * kStageBytes; }
    __device__ __forceinline__ uint32_t w(int s) const { return ring + s * kStageBytes + kXBytes; }
    __device__ __forceinline__ uint32_t vhi() const { return lora; }
    __device__ __forceinline__ uint32_t vlo() const { return lora + kVPart; }
    __device__ __forceinline__ uint32_t bblk(int q) const { return lora + 2 * kVPart + q * RK * 128; }
    __device__ __forceinline__ uint32_t bar(int i) const { return bars + 8 * i; }
  };

  // ------------------------------------------------------------------ TMA producer ----
  __device__ __forceinline__ static void producer(const BaseParams& p, const Smem& sm,
                                                  const Wait& w) {
    if (p.wait_prior_x) pdl_wait_prior();
    int s = 0;
    uint32_t ph = 0, issued = 0, parity = 0;
    for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x) {
      const int m0 = (tile % p.n_mt) * kBM, n0 = (tile / p.n_mt) * kBN;
      for (int kk = 0; kk < p.k_steps; ++kk) {
        if (!w(sm.bar(kEmpty0 + s), ph ^ 1u)) goto out;
        mbar_arrive_expect_tx(sm.bar(kFull0 + s), kStageBytes);
        tma_load_2d(sm.x(s), &p.tmap_x, kk * kBK, m0, sm.bar(kFull0 + s));
        tma_load_2d(sm.w(s), &p.tmap_w, kk * kBK, n0, sm.bar(kFull0 + s));
        issued |= 1u << s;
        parity = (parity & ~(1u << s)) | (ph << s);
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  out:
    sm.ctl[kIssued] = static_cast<int>(issued);
    sm.ctl[kParity] = static_cast<int>(parity);
  }

  // ------------------------------------------------------------------- MMA issuer ----
  __device__ __forceinline__ static void issuer(const BaseParams& p, const Smem& sm,
                                                const Wait& w, uint32_t tm) {
    int s = 0, b = 0;
    uint32_t ph = 0, accph = 0, lph = 0;
    for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x) {
      if (!w(sm.bar(kAccEmpty0 + b), accph ^ 1u)) return;
      tc_fence_after();
      const uint32_t d = tm + static_cast<uint32_t>(b * kBN);
      for (int kk = 0; kk < p.k_steps; ++kk) {
        if (!w(sm.bar(kFull0 + s), ph)) return;
        tc_fence_after();
        const uint32_t xa = sm.x(s), wa = sm.w(s);
#pragma unroll
        for (int j = 0; j < kBK / 16; ++j)
          umma_ss(d, sdesc_sw128(xa + 32u * j, 16, 1024), sdesc_sw128(wa + 32u * j, 16, 1024),
                  kIdBase, (kk | j) != 0);
        umma_commit(sm.bar(kEmpty0 + s));
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      // LoRA rounds: the epilogue posts one message per round, then a closing message
      while (true) {
        if (!w(sm.bar(kLoraFull), lph)) return;
        lph ^= 1u;
        tc_fence_after();
        if (sm.ctl[kCmd] == 0) break;
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int j = 0; j < RK / 16; ++j) {
            const uint64_t bd = sdesc_sw128(sm.bblk(q) + 2048u * j, 8192, 1024);
            umma_ss(d + 64u * q, sdesc_sw128(sm.vhi() + 32u * j, 16, 1024), bd, kIdDelta, 1);
            umma_ss(d + 64u * q, sdesc_sw128(sm.vlo() + 32u * j, 16, 1024), bd, kIdDelta, 1);
          }
        umma_commit(sm.bar(kLoraEmpty));
      }
      umma_commit(sm.bar(kAccFull0 + b));
      if (++b == 2) {
        b = 0;
        accph ^= 1u;
      }
    }
  }

  // --------------------------------------------------------------------- epilogue ----
  // One LoRA round: the operands of adapter k for the tile's rows [m0, m0 + 128) and columns
  // [n0, n0 + 256).  e = epilogue thread index (the row it writes), krow = its row's adapter.
  __device__ __forceinline__ static void build_round(const BaseParams& p, const Smem& sm, int e,
                                                     int t, int krow, int k, int n0) {
    // scale * v of this thread's row (zero for rows of other adapters), split in two parts
    uint32_t hi[RK / 2], lo[RK / 2];
    const bool mine = krow == k;
#pragma unroll
    for (int c = 0; c < RK; c += 4) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (mine && c < p.r) a = __ldg(reinterpret_cast<const float4*>(p.v + static_cast<size_t>(t) * p.r + c));
      const float f[4] = {a.x * p.scale, a.y * p.scale, a.z * p.scale, a.w * p.scale};
      float h[4], l[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        h[u] = round_to<T>(f[u]);
        l[u] = f[u] - h[u];
      }
      hi[c / 2] = pack2<T>(h[0], h[1]);
      hi[c / 2 + 1] = pack2<T>(h[2], h[3]);
      lo[c / 2] = pack2<T>(l[0], l[1]);
      lo[c / 2 + 1] = pack2<T>(l[2], l[3]);
    }
#pragma unroll
    for (int c = 0; c < RK / 8; ++c) {
      sts128(sm.vhi() + sw128(e, c), make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]));
      sts128(sm.vlo() + sw128(e, c), make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]));
    }
    // B_k rows [0, RK) x columns [n0, n0 + 256): rows past r and columns past h_out are zero
    const T* Bk = static_cast<const T*>(p.B_ptrs[k]) + static_cast<size_t>(p.layer) * p.r * p.h_out;
    constexpr int kChunks = RK * 32;  // 16-byte chunks: RK rows x 4 blocks x 8
    for (int u = e; u < kChunks; u += kEpiThreads) {
      const int row = u >> 5, q = (u >> 3) & 3, cc = u & 7;
      const int col = n0 + q * 64 + cc * 8;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (row < p.r && col < p.h_out)
        val = __ldg(reinterpret_cast<const uint4*>(Bk + static_cast<size_t>(row) * p.h_out + col));
      sts128(sm.bblk(q) + sw128(row, cc), val);
    }
    fence_proxy_async();  // generic-proxy writes -> the MMAs' async-proxy reads
  }

  // A wait of the whole epilogue group: one thread waits (bounded) and the group learns the
  // outcome at a named barrier, so that all 128 threads take the same branch afterwards (a
  // thread that left while the others sat at the barrier would hang them).  n: this group
  // wait's sequence number (the result alternates between two words).
  __device__ __forceinline__ static bool group_wait(const Smem& sm, const Wait& w, int e,
                                                    uint32_t bar, uint32_t parity, uint32_t& n) {
    int* slot = sm.ctl + kEpiOk0 + (n & 1u);
    ++n;
    if (e == 0) *reinterpret_cast<volatile int*>(slot) = w(bar, parity) ? 1 : 0;
    named_bar(1, kEpiThreads);
    return *reinterpret_cast<volatile int*>(slot) != 0;
  }

  __device__ __forceinline__ static void epilogue(const BaseParams& p, const Smem& sm,
                                                  const Wait& w, uint32_t tm, int warp) {
    const int lane = threadIdx.x & 31;
    const int qw = warp & 3;                // TMEM lane quarter this warp may read
    const int e = qw * 32 + lane;           // row of the tile
    const uint32_t lane_addr = static_cast<uint32_t>(qw * 32) << 16;
    pdl_wait_prior();  // v is written by the shrink launched just before
    int b = 0;
    uint32_t accph = 0, rounds = 0, nw = 0;
    for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x) {
      const int m0 = (tile % p.n_mt) * kBM, n0 = (tile / p.n_mt) * kBN;
      const int t = m0 + e;
      const int m_end = min(m0 + kBM, p.M);
      int krow = -1;
      if (t < p.M) {
        const int i = segment_of(p.seg_starts, p.S, t);
        if (i >= 0) krow = __ldg(p.seg_adapter + i);
      }
      // the segments that overlap the tile, in order; one round per distinct adapter
      // (segment i overlaps [m0, m_end) iff ss[i] < m_end and ss[i + 1] > m0)
      const int i_lo = max(0, offsets_at_most(p.seg_starts, p.S, m0) - 1);
      const int i_hi = min(p.S - 1, offsets_at_most(p.seg_starts, p.S, m_end - 1) - 1);
      for (int i = i_lo; i <= i_hi; ++i) {
        const int a = max(__ldg(p.seg_starts + i), m0), z = min(__ldg(p.seg_starts + i + 1), m_end);
        const int k = __ldg(p.seg_adapter + i);
        if (z <= a || k < 0) continue;
        bool seen = false;
        for (int j = i_lo; j < i && !seen; ++j) {
          const int aj = max(__ldg(p.seg_starts + j), m0), zj = min(__ldg(p.seg_starts + j + 1), m_end);
          seen = zj > aj && __ldg(p.seg_adapter + j) == k;
        }
        if (seen) continue;
        if (rounds > 0 && !group_wait(sm, w, e, sm.bar(kLoraEmpty), (rounds - 1) & 1u, nw))
          return;
        build_round(p, sm, e, t, krow, k, n0);
        named_bar(1, kEpiThreads);
        if (e == 0) {
          sm.ctl[kCmd] = 1;
          mbar_arrive(sm.bar(kLoraFull));
        }
        ++rounds;
      }
      // closing message (after the last round's operands have been read)
      if (rounds > 0 && !group_wait(sm, w, e, sm.bar(kLoraEmpty), (rounds - 1) & 1u, nw))
        return;
      if (e == 0) {
        sm.ctl[kCmd] = 0;
        mbar_arrive(sm.bar(kLoraFull));
      }
      // the finished tile: TMEM -> output type -> y
      if (!group_wait(sm, w, e, sm.bar(kAccFull0 + b), accph, nw)) return;
      tc_fence_after();
      T* yrow = static_cast<T*>(p.y) + static_cast<size_t>(t) * p.ldy;
#pragma unroll 1
      for (int cc = 0; cc < kBN / 32; ++cc) {
        const int col = n0 + cc * 32;
        if (col >= p.h_out) break;
        uint32_t r[32];
        tmem_ld32(tm + static_cast<uint32_t>(b * kBN + cc * 32) + lane_addr, r);
        tmem_wait_ld();
        if (t < p.M) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (col + 8 * g < p.h_out) {
              const uint4 o = make_uint4(
                  pack2<T>(__uint_as_float(r[8 * g]), __uint_as_float(r[8 * g + 1])),
                  pack2<T>(__uint_as_float(r[8 * g + 2]), __uint_as_float(r[8 * g + 3])),
                  pack2<T>(__uint_as_float(r[8 * g + 4]), __uint_as_float(r[8 * g + 5])),
                  pack2<T>(__uint_as_float(r[8 * g + 6]), __uint_as_float(r[8 * g + 7])));
              *reinterpret_cast<uint4*>(yrow + col + 8 * g) = o;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.bar(kAccEmpty0 + b));
      if (++b == 2) {
        b = 0;
        accph ^= 1u;
      }
    }
  }

  __device__ __forceinline__ static void run(const BaseParams& p) {
    extern __shared__ uint8_t smem_raw[];
    pdl_launch_dependents();
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_addr(smem_raw));
    Smem sm;
    sm.ring = base;
    sm.lora = base + kStages * kStageBytes;
    sm.bars = sm.lora + kLoraBytes;
    sm.ctl = reinterpret_cast<int*>(gbase + kStages * kStageBytes + kLoraBytes + 8 * kNumBars);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
      for (int i = 0; i < kNumCtl; ++i) sm.ctl[i] = 0;
      for (int s = 0; s < kStages; ++s) {
        mbar_init(sm.bar(kFull0 + s), 1);
        mbar_init(sm.bar(kEmpty0 + s), 1);
      }
      mbar_init(sm.bar(kAccFull0), 1);
      mbar_init(sm.bar(kAccFull0 + 1), 1);
      mbar_init(sm.bar(kAccEmpty0), 4);
      mbar_init(sm.bar(kAccEmpty0 + 1), 4);
      mbar_init(sm.bar(kLoraFull), 1);
      mbar_init(sm.bar(kLoraEmpty), 1);
      mbar_init(sm.bar(kDrain), 1);
      mbar_init(sm.bar(kNever), 1);
      fence_mbar_init();
      tma_prefetch_desc(&p.tmap_x);
      tma_prefetch_desc(&p.tmap_w);
    }
    if (warp == 1) {
      tmem_alloc(smem_addr(sm.ctl + kTmem), kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = static_cast<uint32_t>(sm.ctl[kTmem]);
    const Wait w{reinterpret_cast<volatile int*>(sm.ctl + kAbort), p.err, p.wait_ns};
    if (p.inject_stall) w(sm.bar(kNever), 0);  // nothing completes it: the CTA gives up

    if (warp == 0) {
      if (lane_elect()) producer(p, sm, w);
      __syncwarp();
    } else if (warp == 1) {
      if (lane_elect()) {
        issuer(p, sm, w, tm);
        // every MMA this thread issued completes before TMEM is freed
        umma_commit(sm.bar(kDrain));
        w.drain(sm.bar(kDrain), 0);
      }
      __syncwarp();
    } else {
      epilogue(p, sm, w, tm, warp);
    }
    __syncthreads();
    if (sm.ctl[kAbort] && tid == 0) {
      // gave up: the TMA loads still in flight land before the CTA exits
      const uint32_t issued = static_cast<uint32_t>(sm.ctl[kIssued]);
      const uint32_t par = static_cast<uint32_t>(sm.ctl[kParity]);
      for (int s = 0; s < kStages; ++s)
        if ((issued >> s) & 1u) w.drain(sm.bar(kFull0 + s), (par >> s) & 1u);
    }
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tm, kTmemCols);
    }
  }

  __device__ __forceinline__ static bool lane_elect() { return (threadIdx.x & 31) == 0; }
};

template <typename T, int RK>
__global__ void __launch_bounds__(kThreads, 1) base_lora_kernel(const __grid_constant__ BaseParams p) {
  Kernel<T, RK>::run(p);
}

const void* kernel_for(int dtype, int rk) {
  if (dtype == SGMV_F16) {
    if (rk == 16) return reinterpret_cast<const void*>(&base_lora_kernel<__half, 16>);
    if (rk == 32) return reinterpret_cast<const void*>(&base_lora_kernel<__half, 32>);
    if (rk == 64) return reinterpret_cast<const void*>(&base_lora_kernel<__half, 64>);
  } else if (dtype == SGMV_BF16) {
    if (rk == 16) return reinterpret_cast<const void*>(&base_lora_kernel<__nv_bfloat16, 16>);
    if (rk == 32) return reinterpret_cast<const void*>(&base_lora_kernel<__nv_bfloat16, 32>);
    if (rk == 64) return reinterpret_cast<const void*>(&base_lora_kernel<__nv_bfloat16, 64>);
  }
  return nullptr;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeFn>(nullptr);
    return reinterpret_cast<EncodeFn>(f);
  }();
  return fn;
}

// A [rows][cols] 16-bit matrix with row stride ld (elements), boxes of 64 columns x box_rows
// rows, 128-byte swizzle; reads past either extent return zero.
bool encode(Map* out, const void* base, int cols, int rows, int ld, int dtype, int box_rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  CUtensorMap m;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(&m, dtype == SGMV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
         2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  static_assert(sizeof(m) == sizeof(Map), "tensor map size");
  std::memcpy(out, &m, sizeof(m));
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace sgmv_base

extern "C" {

int lora_apply_base(void* y, int32_t ldy, const void* x, int32_t ldx, int32_t M, const void* W0,
                    int32_t ldw, const void* const* A_ptrs, const void* const* B_ptrs,
                    const int32_t* seg_starts, const int32_t* seg_adapter, int32_t num_segments,
                    int32_t layer_idx, int32_t h_in, int32_t h_out, int32_t r, float scale,
                    float* v_work, sgmv_dtype_t dtype, uint32_t flags, sgmv_stream_t stream) {
  using namespace sgmv_base;
  if (M < 0 || num_segments < 0 || layer_idx < 0 || !y || !x || !W0) return SGMV_EINVAL;
  if (flags & ~static_cast<uint32_t>(SGMV_OVERLAP_PRIOR | SGMV_NO_TENSOR_CORES |
                                     SGMV_TENSOR_CORES_ALWAYS | SGMV_LONG_BATCH |
                                     SGMV_DENSE_GRID))
    return SGMV_EINVAL;
  if (dtype != SGMV_F32 && dtype != SGMV_F16 && dtype != SGMV_BF16) return SGMV_EINVAL;
  if (dtype == SGMV_F32) return SGMV_EUNSUPPORTED;  // the tensor cores take 16-bit operands
  if (r != 8 && r != 16 && r != 32 && r != 64) return SGMV_EUNSUPPORTED;
  if (h_in <= 0 || h_out <= 0 || ldx < h_in || ldy < h_out || ldw < h_in) return SGMV_EINVAL;
  if (h_in > SGMV_MAX_HIDDEN || h_out > SGMV_MAX_HIDDEN || ldx > SGMV_MAX_LD ||
      ldy > SGMV_MAX_LD || ldw > SGMV_MAX_LD || num_segments > SGMV_MAX_SEGMENTS)
    return SGMV_EUNSUPPORTED;
  if (h_in % 8 || h_out % 8 || ldx % 8 || ldy % 8 || ldw % 8) return SGMV_EALIGN;
  if (!aligned16(y) || !aligned16(x) || !aligned16(W0)) return SGMV_EALIGN;
  if (num_segments > 0) {
    if (!A_ptrs || !B_ptrs || !seg_starts || !seg_adapter || !v_work) return SGMV_EINVAL;
    if (!aligned16(v_work) || (reinterpret_cast<uintptr_t>(A_ptrs) & 7u) ||
        (reinterpret_cast<uintptr_t>(B_ptrs) & 7u) ||
        (reinterpret_cast<uintptr_t>(seg_starts) & 3u) ||
        (reinterpret_cast<uintptr_t>(seg_adapter) & 3u))
      return SGMV_EALIGN;
  }
  if (M == 0) return SGMV_OK;
  const int rk = r < 16 ? 16 : r;
  const void* fn = kernel_for(dtype, rk);
  if (!fn) return SGMV_EUNSUPPORTED;
  int* err = nullptr;
  int sms = 0, inject = 0;
  uint64_t wait_ns = 0;
  int rc = sgmv::device_context(&err, &sms, &wait_ns, &inject);
  if (rc != SGMV_OK) return rc;

  BaseParams p;
  std::memset(&p, 0, sizeof(p));
  if (!encode(&p.tmap_x, x, h_in, M, ldx, dtype, kBM) ||
      !encode(&p.tmap_w, W0, h_in, h_out, ldw, dtype, kBN))
    return SGMV_ECUDA;
  p.y = y;
  p.v = v_work;
  p.B_ptrs = B_ptrs;
  p.seg_starts = seg_starts;
  p.seg_adapter = seg_adapter;
  p.err = err;
  p.wait_ns = wait_ns;
  p.inject_stall = inject;
  p.S = num_segments;
  p.M = M;
  p.h_in = h_in;
  p.h_out = h_out;
  p.r = r;
  p.layer = layer_idx;
  p.ldy = ldy;
  p.n_mt = (M + kBM - 1) / kBM;
  p.n_tiles = p.n_mt * ((h_out + kBN - 1) / kBN);
  p.k_steps = (h_in + kBK - 1) / kBK;
  p.scale = scale;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // v = x . A_k into the workspace (rows of segments with an adapter); the GEMM below waits
  // for it (programmatic dependent launch) only before its epilogue reads v.
  // The shrink alone streams only x and A: groups of 64 rows and more go to its tensor role
  // (measured at the prefill shape, 4096 -> r = 64, 3450 rows in 8 groups of 142-891 rows:
  // 25 us there against 65 us under the fused call's cost rule, which keeps groups under
  // 256 rows on the CUDA cores), unless the caller turned the tensor cores off.
  const uint32_t shrink_flags =
      (flags & SGMV_NO_TENSOR_CORES) ? flags : (flags | SGMV_TENSOR_CORES_ALWAYS);
  if (num_segments > 0) {
    rc = sgmv_shrink_strided(v_work, x, ldx, A_ptrs, seg_starts, seg_adapter, num_segments,
                             layer_idx, h_in, r, dtype, shrink_flags, stream);
    if (rc != SGMV_OK) return rc;
  }
  // The loads of x may start before the previous kernel has finished only when it is our own
  // shrink launched without SGMV_OVERLAP_PRIOR (then every kernel before it has completed).
  p.wait_prior_x = (flags & SGMV_OVERLAP_PRIOR) ? 1 : 0;
  const bool dependent = num_segments > 0 || (flags & SGMV_OVERLAP_PRIOR);

  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess)
    return SGMV_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(p.n_tiles < sms ? p.n_tiles : sms), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  unsigned na = 0;
  if (dependent) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  void* args[] = {&p};
  return cudaLaunchKernelExC(&cfg, fn, args) == cudaSuccess ? SGMV_OK : SGMV_ECUDA;
}

}  // extern "C"
