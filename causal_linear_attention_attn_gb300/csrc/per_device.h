// A small thread-safe cache of values computed once per (device, key).
//
// CUDA function attributes such as the dynamic shared-memory opt-in belong to
// a device's context, so a launcher that sets one for a kernel must do so
// once on every device it launches on, not once per process.  This table
// keeps one result per (device ordinal, key) pair; the first caller for a
// pair computes it (under the table's lock) and every later caller for the
// same pair gets the stored result.  Plain C++: no CUDA headers, so that the
// logic can be unit-tested on a machine without a GPU.
#pragma once

#include <mutex>
#include <utility>
#include <vector>

namespace la {

template <typename Key, typename Value>
class PerDeviceCache {
 public:
  // The stored value for (dev, key), computing it with make() on first use.
  template <typename Make>
  Value get(int dev, const Key &key, Make &&make) {
    std::lock_guard<std::mutex> lk(mu_);
    for (const Entry &e : entries_)
      if (e.dev == dev && e.key == key) return e.value;
    Value v = make();
    entries_.push_back(Entry{dev, key, v});
    return v;
  }

  // Number of (device, key) pairs computed so far.
  size_t size() {
    std::lock_guard<std::mutex> lk(mu_);
    return entries_.size();
  }

 private:
  struct Entry {
    int dev;
    Key key;
    Value value;
  };
  std::mutex mu_;
  std::vector<Entry> entries_;
};

}  // namespace la
