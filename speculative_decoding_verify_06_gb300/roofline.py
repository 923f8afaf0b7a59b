"""Byte and FLOP accounting of the verify pass (what the roofline fractions divide).

"100 tokens per second ..." (section "The wall") and "Decode is memory-bound ..." (section "The
ceiling") bound decode by bandwidth / bytes read per pass.  Here a pass's algorithmic bytes are
the 4-bit codes and fp16 scales of every real weight (padding excluded), the bf16 activations
read and the fp32 outputs written; nothing dequantised is ever materialised.
"""
from __future__ import annotations

from . import synth


def linear_bytes(in_f: int, out_f: int, C: int) -> int:
    """Algorithmic bytes of one verify-linear launch."""
    return out_f * in_f // 2 + out_f * (in_f // 32) * 2 + C * in_f * 2 + C * out_f * 4


def q4k_linear_bytes(in_f: int, out_f: int, C: int) -> int:
    """Algorithmic bytes of one verify-linear launch on Q4_K weights: 144 bytes per super-block
    of 256 weights (the same 4.5 bits per weight as the symmetric format)."""
    return out_f * (in_f // 256) * 144 + C * in_f * 2 + C * out_f * 4


def linear_weight_bytes(in_f: int, out_f: int) -> int:
    return out_f * in_f // 2 + out_f * (in_f // 32) * 2


def linear_flops(in_f: int, out_f: int, C: int) -> int:
    return 2 * in_f * out_f * C


def stack_bytes(C: int, layers: int = synth.LAYERS) -> int:
    return layers * sum(linear_bytes(i, o, C) for i, o in synth.LAYER_GEMMS)


def stack_weight_bytes(layers: int = synth.LAYERS) -> int:
    return layers * sum(linear_weight_bytes(i, o) for i, o in synth.LAYER_GEMMS)


def stack_flops(C: int, layers: int = synth.LAYERS) -> int:
    return layers * sum(linear_flops(i, o, C) for i, o in synth.LAYER_GEMMS)


def head_bytes(C: int, hidden: int = synth.HIDDEN, vocab: int = synth.VOCAB) -> int:
    """lm_head launch plus the sampler's passes over the logits (S0 and S1 read them, S1 writes
    e, S3 reads e and writes probs)."""
    return linear_bytes(hidden, vocab, C) + C * vocab * 4 * 5


def accept_bytes_per_window(V: int, k: int, rejected: bool) -> int:
    """One vocabulary scan: (p_j, q_j) after a rejection, p_k for the capping draw."""
    return V * 4 * (2 if rejected else 1) + k * 2 * 32


def ceiling(bandwidth_bytes_s: float, bytes_per_pass: float) -> float:
    return bandwidth_bytes_s / bytes_per_pass
