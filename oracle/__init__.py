"""CPU oracle for the NVFP4 MoE expert layer (test infrastructure only)."""
