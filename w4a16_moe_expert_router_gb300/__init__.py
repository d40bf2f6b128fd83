"""W4A16 MoE expert layer for GB300 (sm_103a): C-ABI library binding and synthetic inputs."""
