"""GB300-native FlashAttention-2 forward: a C-ABI CUDA library and its thin binding."""
