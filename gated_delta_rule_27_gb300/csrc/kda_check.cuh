// kda_check.cuh -- bounds checks of libkda's debug build.
//
// Compiled with -DKDA_DEBUG_BOUNDS (libkda_debug.so), every checked index is
// tested before the access it guards: a failed check skips the access and
// records KDA_ERR_BOUNDS in the call's status word, with the source line of
// the first failing check in the word after it, where kda_prefill_check and
// the tests can read them.  The release build (libkda.so) compiles every
// check to `true`.  The checks cover the indices that data decides -- record
// addresses from the chunk table, token rows, state slots -- and the shared
// memory offsets computed from them.
#pragma once

#include <stdint.h>

#include "kda.h"

namespace kda {

#ifdef KDA_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(bool ok, int32_t *status, int line) {
    if (!ok && status) {
        if (atomicCAS(status, 0, (int32_t)KDA_ERR_BOUNDS) == 0) status[1] = line;
    }
    return ok;
}
#define KDA_IN_BOUNDS(cond, status) ::kda::in_bounds((cond), (status), __LINE__)
#else
#define KDA_IN_BOUNDS(cond, status) true
#endif

}  // namespace kda
