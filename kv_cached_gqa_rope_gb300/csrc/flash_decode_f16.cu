// The split-K decode attention (K2 with its combine) for IEEE binary16
// storage: the kernels of flash_decode.cu compiled once more with FP16
// operands.  A translation unit of its own so that both sets compile in
// parallel; its only external symbol is launch_cached_gqa_attention_f16.
#define KVGQA_DECODE_F16 1
#include "flash_decode.cu"
