"""3-D max pooling for GB300 (binding added with the CUDA library)."""
