"""GB300-native context-parallel attention kernels (placeholder: the library
binding lands with the C-ABI)."""
