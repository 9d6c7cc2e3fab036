// Host-only check of the per-context cache the allocation-free build keys its
// table address by (ctx_cache.h): a context id seen before returns its cached
// value without a new lookup, a new id looks the value up again even when an
// earlier context had the same device, a failed lookup caches nothing, and a
// full cache drops its oldest entry.  Exits 0 when every check holds.
#include <cstdio>

#include "ctx_cache.h"

static int fetches = 0;
static char slot_a, slot_b, slot_c;

#define CHECK(c)                                                        \
    do {                                                                \
        if (!(c)) {                                                     \
            std::fprintf(stderr, "check failed line %d: %s\n", __LINE__, #c); \
            return 1;                                                   \
        }                                                               \
    } while (0)

int main()
{
    spc::CtxCache<2> cache;
    auto give = [](void* v) {
        return [v](void** out) {
            ++fetches;
            *out = v;
            return true;
        };
    };
    auto fail = [](void** out) {
        ++fetches;
        *out = nullptr;
        return false;
    };
    CHECK(cache.get(7, give(&slot_a)) == &slot_a);
    CHECK(fetches == 1);
    CHECK(cache.get(7, give(&slot_b)) == &slot_a);  // cached: no second lookup
    CHECK(fetches == 1);
    // a re-created context has a new id and gets its own (new) address
    CHECK(cache.get(8, give(&slot_b)) == &slot_b);
    CHECK(fetches == 2);
    CHECK(cache.get(7, give(&slot_c)) == &slot_a);
    CHECK(fetches == 2);
    // a failed lookup returns nullptr and is not cached
    CHECK(cache.get(9, fail) == nullptr);
    CHECK(fetches == 3);
    CHECK(cache.get(9, give(&slot_c)) == &slot_c);  // evicts id 7, the oldest
    CHECK(fetches == 4);
    CHECK(cache.get(8, give(&slot_a)) == &slot_b);
    CHECK(fetches == 4);
    CHECK(cache.get(7, give(&slot_c)) == &slot_c);  // looked up again
    CHECK(fetches == 5);
    std::puts("ctx cache ok");
    return 0;
}
