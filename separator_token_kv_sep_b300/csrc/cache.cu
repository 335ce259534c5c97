// Streaming cache kernels.  Not built yet: every request reports "not supported".
#include "common.cuh"
#include "layout.h"

#define SEP_API extern "C" __attribute__((visibility("default")))

SEP_API size_t sep_cache_bytes(const sep_cache_params*) { return 0; }
SEP_API sep_status sep_cache_init(const sep_cache_params*, void*, size_t, void*) { return SEP_ERR_UNSUPPORTED; }
SEP_API sep_status sep_cache_step(const sep_cache_params*, void*, const void*, const void*, const void*,
                                  const int32_t*, const int32_t*, int, void*, int, float, void*) { return SEP_ERR_UNSUPPORTED; }
SEP_API size_t sep_cache_export_bytes(const sep_cache_params*) { return 0; }
SEP_API sep_status sep_cache_export(const sep_cache_params*, const void*, void*, size_t, void*) { return SEP_ERR_UNSUPPORTED; }
SEP_API sep_status sep_cache_import(const sep_cache_params*, void*, const void*, size_t, void*) { return SEP_ERR_UNSUPPORTED; }
