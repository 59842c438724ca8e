// tq_attention_generic_d256.cu -- generic attention kernels instantiated for head_dim 256.
#include "tq_attention_generic.cuh"

TQ_ATTENTION_GENERIC_ENTRIES(256)
