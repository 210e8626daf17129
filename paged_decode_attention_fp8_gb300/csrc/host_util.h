// Host-side helpers shared by the launchers (no device code, no CUDA types).
#pragma once

#include <atomic>
#include <cstdint>
#include <utility>

namespace fp8mla {

// Runs `set` for device `dev` unless it already succeeded there: one-time,
// per-device setup such as a kernel's shared-memory limit, which CUDA keeps
// per device.  Bit d of `done` records device d; a device index outside
// [0, 64) runs `set` on every call.  `set` returns a status whose
// value-initialised form ({} : 0 / cudaSuccess) means success; a failure is
// returned and retried on the next call.  Concurrent first calls on one
// device may both run `set`, so it must be idempotent.
template <typename F>
inline auto once_per_device(std::atomic<uint64_t>& done, int dev, F&& set) -> decltype(set()) {
  using Status = decltype(set());
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : uint64_t{0};
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return Status{};
  const Status r = std::forward<F>(set)();
  if (r == Status{} && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return r;
}

}  // namespace fp8mla
