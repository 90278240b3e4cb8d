// checked.cuh -- device-side bounds checks of the library's checked build.
//
// Compiled with -DDGEMM_CHECKED (the build writes libdgemm_checked.so),
// DGEMM_CHECK(cond) evaluates a condition on an index a kernel computed -- a
// shared-memory offset, a tile coordinate, a global row or column, the
// alignment a vector access needs -- against the extent it must stay inside.
// A failed check records DGEMM_ERR_BOUNDS and the site (this translation
// unit's number x 100000 + the source line) in the unit's check words, and
// the caller skips the access the check guards: nothing traps, no access
// goes out of bounds, and the kernel runs to its end.  The first failure
// since the last clear is the one kept.  In the normal build DGEMM_CHECK is
// the constant true and compiles away.
//
// Device code is not linked across translation units, so each unit that
// includes this header has its own check words and defines its own reader
// (DGEMM_DEFINE_CHECK_READER), which dgemm_device_status and
// dgemm_check_site combine.
#pragma once

#include <cuda_runtime.h>

#include "dgemm.h"

#ifndef DGEMM_UNIT
#error "define DGEMM_UNIT (this translation unit's number) before including checked.cuh"
#endif

namespace dgemm {
namespace {

#ifdef DGEMM_CHECKED
__device__ int g_check_status;  // DGEMM_ERR_BOUNDS once a check has failed
__device__ int g_check_site;    // site of the first failed check

__device__ __forceinline__ bool check_passed(bool ok, int site)
{
    if (!ok && atomicCAS(&g_check_status, 0, DGEMM_ERR_BOUNDS) == 0) atomicExch(&g_check_site, site);
    return ok;
}

#define DGEMM_CHECK(cond) (::dgemm::check_passed(static_cast<bool>(cond), DGEMM_UNIT * 100000 + __LINE__))
// The same check, answered for the whole CTA (true only if it passed in every
// thread), for decisions that barriers depend on.  Every thread of the CTA
// must reach it.
#define DGEMM_CHECK_CTA(cond) (__syncthreads_and(DGEMM_CHECK(cond) ? 1 : 0) != 0)

// This unit's check words: the status (0 or DGEMM_ERR_BOUNDS) is returned,
// the site written to *site; both are reset when clear != 0.
int read_check_words(int clear, int *site)
{
    int st = 0, where = 0;
    if (cudaMemcpyFromSymbol(&st, g_check_status, sizeof(int)) != cudaSuccess ||
        cudaMemcpyFromSymbol(&where, g_check_site, sizeof(int)) != cudaSuccess)
        return DGEMM_ERR_LAUNCH;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_check_status, &zero, sizeof(int)) != cudaSuccess ||
            cudaMemcpyToSymbol(g_check_site, &zero, sizeof(int)) != cudaSuccess)
            return DGEMM_ERR_LAUNCH;
    }
    if (site) *site = where;
    return st;
}
#else
#define DGEMM_CHECK(cond) true
#define DGEMM_CHECK_CTA(cond) true

int read_check_words(int, int *site)
{
    if (site) *site = 0;
    return 0;
}
#endif

}  // namespace
}  // namespace dgemm

// Defines `int name(int clear, int *site)` in namespace dgemm: this unit's
// check words (declared in internal.h).
#define DGEMM_DEFINE_CHECK_READER(name)                  \
    namespace dgemm {                                    \
    int name(int clear, int *site)                       \
    {                                                    \
        return read_check_words(clear, site);            \
    }                                                    \
    }
