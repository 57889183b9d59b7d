// Encode dispatch: the kernels for each key width are compiled in their own
// translation unit (tq_inst.cu, built once per width).
#include <cuda_runtime.h>

#include "tq_internal.h"

namespace tq {

int launch_encode(const EncodeArgs& a, int num_sms, void* stream) {
    switch (a.g.kb) {
        case 1: return launch_encode_kb<1>(a, num_sms, stream);
        case 2: return launch_encode_kb<2>(a, num_sms, stream);
        case 3: return launch_encode_kb<3>(a, num_sms, stream);
        case 4: return launch_encode_kb<4>(a, num_sms, stream);
        case 5: return launch_encode_kb<5>(a, num_sms, stream);
        case 6: return launch_encode_kb<6>(a, num_sms, stream);
        case 7: return launch_encode_kb<7>(a, num_sms, stream);
        case 8: return launch_encode_kb<8>(a, num_sms, stream);
        default: return (int)cudaErrorInvalidValue;
    }
}

}  // namespace tq
