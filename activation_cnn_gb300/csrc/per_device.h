// per_device.h -- bookkeeping of one-time, per-device actions on the host.
//
// Some CUDA settings act on the current device only (a kernel's dynamic
// shared-memory opt-in, cudaFuncSetAttribute): a process that drives several
// GPUs must apply them on each.  PerDeviceSizes records, for each (key,
// device) pair, the largest size an action was applied with; an action is
// needed again when a larger size is asked for, or on another device.
// Thread-safe; plain C++ (no CUDA), so it is tested on the host alone.
#pragma once

#include <cstddef>
#include <mutex>
#include <vector>

namespace acnn {

class PerDeviceSizes {
public:
    // Run apply() (returning true on success) unless (key, dev) already
    // holds a size >= bytes; on success record bytes.  Returns false only
    // when apply() was needed and failed.  apply() runs under the lock.
    template <typename F> bool ensure(const void* key, int dev, size_t bytes, F&& apply) {
        std::lock_guard<std::mutex> lk(mu_);
        for (Entry& e : entries_)
            if (e.key == key && e.dev == dev) {
                if (e.bytes >= bytes) return true;
                if (!apply()) return false;
                e.bytes = bytes;
                return true;
            }
        if (!apply()) return false;
        entries_.push_back(Entry{key, dev, bytes});
        return true;
    }

private:
    struct Entry {
        const void* key;
        int dev;
        size_t bytes;
    };
    std::mutex mu_;
    std::vector<Entry> entries_;
};

}  // namespace acnn
