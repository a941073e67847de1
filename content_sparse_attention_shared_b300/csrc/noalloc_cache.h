// Host-side cache for rt_route_assign_noalloc: the device addresses of the
// library's fixed scratch array and status word, per CUDA context.
//
// A file-scope __device__ array has one instance per context that loads the
// module, at an address that is only valid in that context.  The cache is
// therefore keyed on the context's unique id (cuCtxGetId), not on the device
// number: after a device reset, or in a second context on the same device,
// the id differs, the lookup misses and the caller asks the runtime for the
// address again instead of reusing a stale one.  Plain C++, no CUDA calls, so
// the key logic is testable on a machine without a GPU.
#pragma once

namespace rt {

struct NoallocAddrs {
  void* scores = nullptr;
  void* status = nullptr;
};

template <int N>
class ContextAddressCache {
 public:
  // The entry of context `id`, or nullptr.
  const NoallocAddrs* find(unsigned long long id) const {
    for (int i = 0; i < used_; ++i)
      if (ids_[i] == id) return &addrs_[i];
    return nullptr;
  }
  // Records (or replaces) the entry of context `id`; when full, the oldest
  // entry is dropped.
  void put(unsigned long long id, const NoallocAddrs& a) {
    for (int i = 0; i < used_; ++i)
      if (ids_[i] == id) {
        addrs_[i] = a;
        return;
      }
    ids_[next_] = id;
    addrs_[next_] = a;
    next_ = (next_ + 1) % N;
    if (used_ < N) ++used_;
  }
  int size() const { return used_; }

 private:
  unsigned long long ids_[N] = {};
  NoallocAddrs addrs_[N];
  int used_ = 0, next_ = 0;
};

}  // namespace rt
