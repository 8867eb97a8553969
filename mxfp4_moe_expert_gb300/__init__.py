"""MXFP4 MoE expert layer for GB300 (sm_103a): Python binding of the C ABI."""
