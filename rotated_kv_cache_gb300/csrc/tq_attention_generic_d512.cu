// tq_attention_generic_d512.cu -- generic attention kernels instantiated for head_dim 512.
#include "tq_attention_generic.cuh"

TQ_ATTENTION_GENERIC_ENTRIES(512)
