// Batch-pair kernels specialised for one layer shape (see wtconv_pair_specs.h).
#include "wtconv_pair_fwd.cuh"
#include "wtconv_pair_specs.h"

namespace wtconv {
WTCONV_CALL(WTCONV_PAIR_SPEC_DEF, WTCONV_SPEC_b64l4)
}  // namespace wtconv
