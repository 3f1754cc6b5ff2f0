// decode_inst_3.cu -- explicit instantiations (group 3) of the decode kernel; see decode_instances.inc.
#include "decode_kernel.cuh"
#define KVQ_GROUP 3
#define KVQ_X(KF, VF, PKF, PVF, NW) KVQ_DECODE_INSTANCE(KF, VF, PKF, PVF, NW, false) KVQ_DECODE_INSTANCE(KF, VF, PKF, PVF, NW, true)
#include "decode_instances.inc"
