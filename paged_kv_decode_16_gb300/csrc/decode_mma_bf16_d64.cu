// decode_mma_bf16_d64.cu -- bf16, head_dim 64 instantiations of the tensor-core decode kernel.
#include "decode_mma.cuh"

namespace pkv {

DecodeMmaInfo decode_mma_info_bf16_d64(int gs) {
    using T = __nv_bfloat16;
    switch (gs) {
        case 1: return make_decode_mma_info<T, 64, 1>();
        case 2: return make_decode_mma_info<T, 64, 2>();
        case 3: return make_decode_mma_info<T, 64, 3>();
        case 4: return make_decode_mma_info<T, 64, 4>();
        case 5: return make_decode_mma_info<T, 64, 5>();
        case 6: return make_decode_mma_info<T, 64, 6>();
        case 7: return make_decode_mma_info<T, 64, 7>();
        case 8: return make_decode_mma_info<T, 64, 8>();
        case 9: return make_decode_mma_info<T, 64, 9>();
        case 10: return make_decode_mma_info<T, 64, 10>();
        case 11: return make_decode_mma_info<T, 64, 11>();
        case 12: return make_decode_mma_info<T, 64, 12>();
        case 13: return make_decode_mma_info<T, 64, 13>();
        case 14: return make_decode_mma_info<T, 64, 14>();
        case 15: return make_decode_mma_info<T, 64, 15>();
        case 16: return make_decode_mma_info<T, 64, 16>();
        case 32: return make_decode_mma_info<T, 64, 32>();  // two tiles of 16 rows
    }
    return DecodeMmaInfo{nullptr, 0, 0, 0, 0};
}

}  // namespace pkv
