"""GB300-native paged GQA decode attention (CUDA library + thin Python binding)."""
