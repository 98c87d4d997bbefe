"""Layer-by-layer parity against the oracle, shared by the decode, prefill and batch tests (test support)."""
import numpy as np

import oracle


def rel_err(gpu, ora):
    gpu = np.asarray(gpu, np.float64)
    ora = np.asarray(ora, np.float64)
    return float(np.max(np.abs(gpu - ora)) / max(np.max(np.abs(ora)), 1e-300))


def layer_vs_oracle(mode, om, l, pos, h_in, h_out, tol):
    """Layer l of the oracle from the GPU's input row h_in, against the GPU's output row h_out (the row and its
    increment).  In the one-word mode each word of an activation decides by rounding x/d; where that value lies within
    1e-4 of a step of a rounding boundary, the GPU (whose input to the rule differs from the oracle's in its last bits)
    may round it the other way, and both words are results of the rule.  When the oracle's own result misses the
    tolerance, the results with such words rounded the other way (one or two of the four nearest a boundary) are tried:
    the words of the attention output the O projection reads, then those of the mixture's input.
    Returns (router logits, error of the matching result, (site, word) rounded the other way or None)."""
    def err(h_ora):
        return max(rel_err(h_out, h_ora), rel_err(h_out.astype(np.float64) - h_in, h_ora.astype(np.float64) - h_in))
    h_ora, rl = oracle.decode_layer(mode, om, l, pos, h_in)
    e = err(h_ora)
    if e < tol or mode != 1:
        return rl, e, None
    for site in (oracle.PROBE_ATTN_OUT, oracle.PROBE_MOE_INPUT):
        _, _, mg = oracle.decode_layer(mode, om, l, pos, h_in, probe=True, site=site)
        # the other rounding of each word on a boundary (an exact tie's margin is a signed zero: its sign still
        # points to the other rounding), alone and in pairs
        near = [(int(i), -1 if np.signbit(mg[i]) else 1) for i in np.argsort(np.abs(mg))[:4] if abs(mg[i]) < 1e-4]
        for flips in [[f] for f in near] + [[a, b] for j, a in enumerate(near) for b in near[j + 1:]]:
            h_alt, _ = oracle.decode_layer(mode, om, l, pos, h_in, flips=flips, site=site)
            if err(h_alt) < tol:
                return rl, err(h_alt), (site, [i for i, _ in flips])
    return rl, e, None
