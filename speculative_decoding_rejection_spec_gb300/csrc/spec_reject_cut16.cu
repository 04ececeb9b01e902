// The first-rejection pass with top-k / top-p cuts, built with 16 warps per block (one block per
// SM) from the same source: every reached row's cut runs on twice the warps, which shortens each
// request's chain of rows where a batch does not fill the GPU with 8-warp blocks.  The library's
// dispatch (spec_reject.cu) picks it by batch size.
#define SPEC_KL_WARPS 16
#define SPEC_KL_MIN_BLOCKS 1
#define SPEC_KL_CUT_VARIANT 1
#include "spec_reject.cu"
