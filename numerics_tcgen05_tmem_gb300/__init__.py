"""GB300-native stabilised FlashAttention: C-ABI CUDA library and its Python binding."""
