"""fp64 CPU oracle (test infrastructure; never imported by the product path)."""
from .attn_ref import backward, forward, head_backward, head_forward, kv_head, scores

__all__ = ["backward", "forward", "head_backward", "head_forward", "kv_head", "scores"]
