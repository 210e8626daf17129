// Shared constants and the bounded mbarrier wait used by every kernel.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>
#include <utility>

#include "fp8mla.h"
#include "host_util.h"
#include "ptx.cuh"

namespace fp8mla {

// The last N tensor maps an entry point encoded, by (base pointer, extent,
// device): a map depends on nothing else (its boxes and strides are fixed per
// entry point), so a call on the same cache skips the host-side encoding.
template <int N>
class TensorMapCache {
 public:
  template <typename Encode>
  bool get(const void* base, long long extent, CUtensorMap* out, Encode&& encode) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu_);
    for (const Entry& e : entries_)
      if (e.used && e.base == base && e.extent == extent && e.device == dev) {
        *out = e.map;
        return true;
      }
    CUtensorMap m;
    if (!encode(&m)) return false;
    entries_[next_] = Entry{base, extent, dev, true, m};
    next_ = (next_ + 1) % N;
    *out = m;
    return true;
  }

 private:
  struct Entry {
    const void* base;
    long long extent;
    int device;
    bool used;
    CUtensorMap map;
  };
  std::mutex mu_;
  Entry entries_[N] = {};
  int next_ = 0;
};

// A wait that has not completed after this long is treated as a hang: the
// kernel records FP8MLA_DEV_WAIT_TIMEOUT and stops instead of spinning on.
// The limit lives in device memory (one copy per translation unit) so that a
// test can shorten it for the kernels of one file (fp8mla_test_fault_injection).
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr uint32_t kWaitMinPolls = 1u << 16;
static __device__ uint64_t g_wait_limit_ns = kWaitLimitNs;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

// The first bounded wait of this translation unit's kernels that ran out:
// {site (a source line), block, thread, recorded}; read and cleared by the host.
static __device__ uint32_t g_timeout_where[4];

__device__ __forceinline__ void record_timeout_site(uint32_t site) {
  if (atomicCAS(&g_timeout_where[3], 0u, 1u) == 0u) {
    g_timeout_where[0] = site;
    g_timeout_where[1] = blockIdx.x;
    g_timeout_where[2] = threadIdx.x;
  }
}

// Bounded wait on an mbarrier phase.  Returns false (without waiting further)
// once *abort_flag is set by any thread of the CTA, or after the limit, in
// which case it sets the flag and the status bit itself.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                             uint32_t* status, uint32_t site = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (it > kWaitMinPolls && globaltimer_ns() - t0 > *(volatile uint64_t*)&g_wait_limit_ns) {
        if (abort_flag != nullptr) *abort_flag = 1u;
        atomicOr(status, FP8MLA_DEV_WAIT_TIMEOUT);
        record_timeout_site(site);
        return false;
      }
    }
  }
}

// The same contract as wait_bounded, but polling with the non-blocking probe:
// for waits on the critical path, where a suspended thread wakes up late.
__device__ __forceinline__ bool wait_spin(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint32_t* status, uint32_t site = 0) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (it > kWaitMinPolls && globaltimer_ns() - t0 > *(volatile uint64_t*)&g_wait_limit_ns) {
        if (abort_flag != nullptr) *abort_flag = 1u;
        atomicOr(status, FP8MLA_DEV_WAIT_TIMEOUT);
        record_timeout_site(site);
        return false;
      }
    }
  }
}

// Pages of a sequence; 0 (and a status bit) for a length the block table cannot hold.
__device__ __forceinline__ int seq_pages(int s_k, int page, int max_pages, uint32_t* status) {
  if (s_k <= 0) {
    if (s_k < 0) atomicOr(status, FP8MLA_DEV_BAD_SEQLEN);
    return 0;
  }
  const int n = (s_k + page - 1) / page;
  if (n > max_pages) {
    atomicOr(status, FP8MLA_DEV_BAD_SEQLEN);
    return 0;
  }
  return n;
}

// One arrival per warp: every lane's earlier work (shared-memory writes,
// completed tcgen05 loads/stores followed by tcgen05.fence::before_thread_sync)
// is ordered before lane 0's release-arrive by the warp barrier.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// once_per_device on the current device; a failing cudaGetDevice is returned.
template <typename F>
inline cudaError_t configure_once(std::atomic<uint64_t>& done, F&& set) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return once_per_device(done, dev, std::forward<F>(set));
}

// Launches `kernel` on `stream` as a programmatic dependent of the previous
// work in the stream: its CTAs may start while that work finishes, so the
// kernel must call griddep_wait() before touching memory the predecessor
// writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace fp8mla
