// cfgstep_internal.h -- declarations shared by the library's translation units
// (not part of the C ABI; every symbol here has hidden visibility).
#ifndef CFGSTEP_INTERNAL_H
#define CFGSTEP_INTERNAL_H

#include <cuda_runtime.h>

namespace cfgstep {

// Record a printf-style message for cfg_last_error() on this host thread and
// return `code`.
int fail(int code, const char* fmt, ...);
// fail(CFG_ERR_CUDA, ...) with the CUDA runtime's name and text of `e`.
int cuda_fail(cudaError_t e, const char* what);

}  // namespace cfgstep

#endif  // CFGSTEP_INTERNAL_H
