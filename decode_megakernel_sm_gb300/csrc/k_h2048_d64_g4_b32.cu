#include "megakernel.cuh"

namespace mk {
extern const Variant variant_h2048_d64_g4_b32 = {2048, 64, 4, 32, 2,
                                               (const void*)&mk_decode_kernel<2048, 64, 4, 32, 2>};
}  // namespace mk
