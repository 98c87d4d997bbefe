// Regions of device memory a kernel asks L2 to fetch ahead of their use (weights of later launches of the step).
#pragma once
#include <stddef.h>

namespace q8 {

struct L2Prefetch {
    static constexpr int kMax = 6;
    const void* ptr[kMax] = {};
    size_t bytes[kMax] = {};
    int n = 0;
    void add(const void* p, size_t b) {
        if (p && b && n < kMax) {
            ptr[n] = p;
            bytes[n] = b;
            ++n;
        }
    }
};

}  // namespace q8
