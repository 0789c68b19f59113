"""OCP-MX block quantization (MXFP4 / MXFP8) for GB300."""
