"""GB300-native int4 gathered-expert MoE block (Edge0 streaming-MoE hot path).

Importing the package loads nothing; ``int4_gathered_expert_gb300.lib`` loads
the CUDA library (and fails loudly when it is missing).
"""
__all__ = ["synth"]
