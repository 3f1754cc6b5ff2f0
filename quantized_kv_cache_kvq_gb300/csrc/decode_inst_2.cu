// decode_inst_2.cu -- explicit instantiations (group 2) of the decode kernel; see decode_instances.inc.
#include "decode_kernel.cuh"
#define KVQ_GROUP 2
#define KVQ_X(KF, VF, PKF, PVF, NW) KVQ_DECODE_INSTANCES(KF, VF, PKF, PVF, NW)
#include "decode_instances.inc"
// the INT8-dithered layout with the fixed-channel key outlier bypass
KVQ_DECODE_INSTANCES3(KVQ_FMT_INT8_DITHER, KVQ_FMT_INT8_DITHER, -1, -1, 12, true)
