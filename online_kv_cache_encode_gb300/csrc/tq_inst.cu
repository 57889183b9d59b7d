// The encode and decode kernels of one key width, TQ_KB (1 .. 8), with every
// value width.  The build compiles this file once per key width.
#include "tq_decode_impl.cuh"
#include "tq_encode_impl.cuh"

#ifndef TQ_KB
#error "compile with -DTQ_KB=<key width>"
#endif

namespace tq {
template int launch_encode_kb<TQ_KB>(const EncodeArgs&, int, void*);
template int launch_decode_kb<TQ_KB>(const DecodeArgs&, void*);
template int decode_smem_kb<TQ_KB>(const Geometry&);
}  // namespace tq
