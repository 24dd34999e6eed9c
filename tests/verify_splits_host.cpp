// Host-only driver of the verify kernel's split plans (masw_splits.h): prints
// "pairs NQ Tmax slots plan noalloc" for a grid of shapes and resident-slot
// counts, with D = 128, at most 64 splits and the 4 MiB cap of the
// allocation-free entry point.  Run by test_verify_splits_host.py.
#include <cstdio>

#include "../compressed_draft_kv_gb300/csrc/masw_splits.h"

int main() {
    const int pairs[] = {1, 2, 3, 5, 8, 16, 32, 64, 100, 152, 256, 1000, 4096};
    const int nqs[] = {1, 4, 8, 16, 24, 32};
    const int tmaxs[] = {256, 1000, 32768};
    const int slots[] = {152, 304, 1024, 4096};
    const size_t cap = (size_t)4 << 20;
    for (int pr : pairs)
        for (int nq : nqs)
            for (int tm : tmaxs)
                for (int sl : slots)
                    std::printf("%d %d %d %d %d %d\n", pr, nq, tm, sl, masw::verify_split_plan(pr, sl, tm, 64),
                                masw::noalloc_split_plan(pr, nq, 128, tm, sl, 64, cap));
    return 0;
}
