// decode_inst_1.cu -- explicit instantiations (group 1) of the decode kernel; see decode_instances.inc.
#include "decode_kernel.cuh"
#define KVQ_GROUP 1
#define KVQ_X(KF, VF, PKF, PVF, NW) KVQ_DECODE_INSTANCES(KF, VF, PKF, PVF, NW)
#include "decode_instances.inc"
