// tq_attention_generic_d64.cu -- generic attention kernels instantiated for head_dim 64.
#include "tq_attention_generic.cuh"

TQ_ATTENTION_GENERIC_ENTRIES(64)
