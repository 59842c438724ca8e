// tq_attention_generic_d128.cu -- generic attention kernels instantiated for head_dim 128.
#include "tq_attention_generic.cuh"

TQ_ATTENTION_GENERIC_ENTRIES(128)
