"""CPU oracle for the K3 LatentMoE routed-expert layer (test infrastructure only)."""
