"""GB300-native PagedAttention decode: paged K/V cache kernels behind a C ABI."""
