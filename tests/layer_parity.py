"""Layer-by-layer parity against the oracle, shared by the decode, prefill and batch tests (test support)."""
import numpy as np

import oracle


def rel_err(gpu, ora):
    gpu = np.asarray(gpu, np.float64)
    ora = np.asarray(ora, np.float64)
    return float(np.max(np.abs(gpu - ora)) / max(np.max(np.abs(ora)), 1e-300))


def check_token(gpu_tok, ora_logits, tol):
    """The greedy token against the oracle's logits.  Logits within the mode's tolerance (relative to the largest
    magnitude) fix the arg-max only when the oracle's top two differ by more than twice that bound; inside the band
    either of the close candidates is a correct result, so the GPU's token must then be one of them (its oracle logit
    within the band of the top)."""
    ora_logits = np.asarray(ora_logits, np.float64)
    band = 2.0 * tol * float(np.max(np.abs(ora_logits)))
    srt = np.sort(ora_logits)[::-1]
    if srt[0] - srt[1] > band:
        assert int(gpu_tok) == int(np.argmax(ora_logits)), (int(gpu_tok), int(np.argmax(ora_logits)))
    else:
        assert ora_logits[int(gpu_tok)] >= srt[0] - band, (int(gpu_tok), ora_logits[int(gpu_tok)], srt[0], band)


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
