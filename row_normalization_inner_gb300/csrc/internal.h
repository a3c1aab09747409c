// Entry-point internals shared between the C ABI translation units.
#pragma once

#include "../../include/nf.h"

namespace nf {

// The LayerNorm backward behind nf_layernorm_bwd and
// nf_layernorm_bwd_noalloc.  With `scratch` null it is nf_layernorm_bwd.
// With `scratch` set, the workspace is a fixed area of `workspace_bytes`
// bytes owned by the library: `workspace` is ignored, every argument is
// checked first, a plan whose partials need more than the area returns
// NF_ERR_WORKSPACE_TOO_SMALL, and only then is the area's address fetched
// with scratch().
nf_status layernorm_bwd_impl(void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                             const float* mean, const float* rstd, const void* gamma, int64_t rows,
                             int64_t hidden, void* workspace, size_t workspace_bytes,
                             nf_status (*scratch)(void**), nf_stream stream);

}  // namespace nf
