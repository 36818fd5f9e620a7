"""GB300-native active-expert-chunked low-precision MoE layer with a
block-diagonal orthogonal adapter (see ``include/pmoe.h`` for the C ABI)."""
