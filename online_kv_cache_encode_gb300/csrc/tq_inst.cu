// The encode and decode kernels of one key width, TQ_KB (1 .. 8), with every
// value width.  The build compiles this file once per key width.
#include "tq_decode_impl.cuh"
#include "tq_encode_impl.cuh"
#if TQ_KB == 4
#include "tq_decode_tc.cuh"
#endif

#ifndef TQ_KB
#error "compile with -DTQ_KB=<key width>"
#endif

namespace tq {
template int launch_encode_kb<TQ_KB>(const EncodeArgs&, int, void*);
template int launch_decode_kb<TQ_KB>(const DecodeArgs&, void*);
template int decode_smem_kb<TQ_KB>(const Geometry&);
#if TQ_KB == 4
int launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
    switch (a.g.vb) {
        case 1: return launch_decode_tc_t<1>(a, s);
        case 2: return launch_decode_tc_t<2>(a, s);
        case 3: return launch_decode_tc_t<3>(a, s);
        case 4: return launch_decode_tc_t<4>(a, s);
        default: return (int)cudaErrorNotSupported;
    }
}
#endif
}  // namespace tq
