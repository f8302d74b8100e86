// One compiled instantiation of the decode interpreter: hidden 2048, head_dim 64,
// 4 query heads per kv head, batch capacity 8.
#include "megakernel.cuh"

namespace mk {
extern const Variant variant_h2048_d64_g4_b8 = {2048, 64, 4, 8, 2,
                                              (const void*)&mk_decode_kernel<2048, 64, 4, 8, 2>};
}  // namespace mk
