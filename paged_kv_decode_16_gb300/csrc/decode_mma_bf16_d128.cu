// decode_mma_bf16_d128.cu -- bf16, head_dim 128 instantiations of the tensor-core decode kernel.
#include "decode_mma.cuh"

namespace pkv {

DecodeMmaInfo decode_mma_info_bf16_d128(int gs) {
    using T = __nv_bfloat16;
    switch (gs) {
        case 1: return make_decode_mma_info<T, 128, 1>();
        case 2: return make_decode_mma_info<T, 128, 2>();
        case 3: return make_decode_mma_info<T, 128, 3>();
        case 4: return make_decode_mma_info<T, 128, 4>();
        case 5: return make_decode_mma_info<T, 128, 5>();
        case 6: return make_decode_mma_info<T, 128, 6>();
        case 7: return make_decode_mma_info<T, 128, 7>();
        case 8: return make_decode_mma_info<T, 128, 8>();
        case 9: return make_decode_mma_info<T, 128, 9>();
        case 10: return make_decode_mma_info<T, 128, 10>();
        case 11: return make_decode_mma_info<T, 128, 11>();
        case 12: return make_decode_mma_info<T, 128, 12>();
        case 13: return make_decode_mma_info<T, 128, 13>();
        case 14: return make_decode_mma_info<T, 128, 14>();
        case 15: return make_decode_mma_info<T, 128, 15>();
        case 16: return make_decode_mma_info<T, 128, 16>();
        case 32: return make_decode_mma_info<T, 128, 32>();  // two tiles of 16 rows
    }
    return DecodeMmaInfo{nullptr, 0, 0, 0, 0};
}

}  // namespace pkv
