// ctx_cache.h -- a small fixed-size cache of one value per CUDA context, keyed
// by the context's unique id (cuCtxGetId: ids are never reused within a
// process, unlike context handles, which a reset or a new context can repeat).
// Plain C++ with no CUDA dependency, so its logic is testable on any host.
#pragma once

#include <mutex>
#include <stdint.h>

namespace spc {

template <int N>
class CtxCache {
public:
    // The value cached for context `id`, or the one `fetch(&v)` produces (it
    // returns true on success) and is then cached; nullptr when fetch fails.
    // When the cache is full the oldest entry gives way.
    template <typename Fetch>
    void* get(unsigned long long id, Fetch fetch)
    {
        std::lock_guard<std::mutex> guard(lock_);
        for (int i = 0; i < used_; ++i)
            if (ids_[i] == id) return vals_[i];
        void* v = nullptr;
        if (!fetch(&v) || !v) return nullptr;
        ids_[next_] = id;
        vals_[next_] = v;
        next_ = (next_ + 1) % N;
        if (used_ < N) ++used_;
        return v;
    }

private:
    std::mutex lock_;
    unsigned long long ids_[N] = {};
    void* vals_[N] = {};
    int used_ = 0, next_ = 0;
};

}  // namespace spc
