// Key-split plans of the verify kernel, as plain host functions (no CUDA), so
// that the allocation-free entry point's reduction -- which no shape reaches on
// a 152-SM GB300 -- can be checked on the host with larger SM counts.
#pragma once

#include <stddef.h>

#include <algorithm>

namespace masw {

// Splits per (sequence, kv head) pair: one wave of the `slots` resident CTA
// slots over `pairs` pairs, at least 256 keys per split, at most max_split.
inline int verify_split_plan(int pairs, int slots, int Tmax, int max_split) {
    int n = std::max(1, slots / std::max(1, pairs));
    n = std::min(n, std::max(1, (Tmax + 255) / 256));
    return std::min(n, max_split);
}

// Bytes of the split partials: per pair and split, NQ query rows of D outputs
// plus the row max and sum (floats), rounded up to 256 bytes.
inline size_t verify_partial_bytes(int pairs, int NQ, int D, int n_split) {
    const size_t b = (size_t)pairs * n_split * NQ * (D + 2) * sizeof(float);
    return ((b + 255) / 256) * 256;
}

// The allocation-free entry point's split count: the usual plan, lowered until
// the partials fit in `cap` bytes.  One split writes no partials (its CTA
// stores the output itself), so the result always fits.  With one CTA per SM
// the plan's partials take at most slots * NQ * (D + 2) * 4 bytes, which is
// below a 4 MiB cap up to about 250 SMs: the reduction is reached only on
// larger devices or with more resident CTAs per SM.
inline int noalloc_split_plan(int pairs, int NQ, int D, int Tmax, int slots, int max_split, size_t cap) {
    int n = verify_split_plan(pairs, slots, Tmax, max_split);
    while (n > 1 && verify_partial_bytes(pairs, NQ, D, n) > cap) --n;
    return n;
}

}  // namespace masw
