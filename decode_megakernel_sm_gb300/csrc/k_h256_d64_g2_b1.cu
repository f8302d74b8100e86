// One compiled instantiation of the decode interpreter: hidden 256, head_dim 64,
// 2 query heads per kv head, batch capacity 1.
#include "megakernel.cuh"

namespace mk {
extern const Variant variant_h256_d64_g2_b1 = {256, 64, 2, 1, 2,
                                              (const void*)&mk_decode_kernel<256, 64, 2, 1, 2>};
}  // namespace mk
