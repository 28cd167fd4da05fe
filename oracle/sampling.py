"""CPU oracle of the decode step's token choice when it samples instead of taking the argmax.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's CPU baseline
leg may import this module.  The engine never does; the two share no code.

What it computes, in plain float64 (the pages fix no precision for the sampler):
  * temperature <= 0: greedy, the argmax of the logits (lowest index on ties)
    ["FlashQwen", "Stage 5 - GPU argmax for greedy"];
  * otherwise ["FlashQwen", run options --temperature / --top-k / --top-p, Qwen's recommended
    0.6 / 20 / 0.95; naive Qwen engine, "Sampler": Top-K draws among the k most probable]:
      1. the k largest logits, ties broken by the lowest index, in decreasing order;
      2. weights w_i = exp((l_i - l_0) / temperature) (l_0 the largest; the softmax of
         logits / temperature up to its normaliser);
      3. top-p: the smallest prefix 0..n of them whose weight reaches top_p of their sum;
      4. u uniform in [0, 1) from the counter-based generator below; the token is the first
         index j of the prefix whose running sum exceeds u times the prefix's sum.
    Reading (the pages do not order the filters): top-k, then top-p on the renormalised k.

Generator: SplitMix64 (Steele, Lea & Flood, OOPSLA 2014; the published sequential form
`state += 0x9E3779B97F4A7C15; return mix(state)`), started at mix(seed); draw number `counter`
is mix(mix(seed) + (counter + 1) * 0x9E3779B97F4A7C15), and u is its top 24 bits * 2^-24 (exact
in float32).  The engine draws with counter = the position whose logits are sampled.
"""
import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MASK = (1 << 64) - 1


def mix(z):
    """The SplitMix64 output mix (Vigna's constants)."""
    z &= MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def uniform(seed, counter):
    """u in [0, 1) with 24 significant bits, a pure function of (seed, counter)."""
    x = mix(mix(seed) + (counter + 1) * GAMMA)
    return (x >> 40) * 2.0 ** -24


def sample(logits, temperature, top_k, top_p, seed, counter):
    """Returns (token, kept, margin): the drawn token, the indices of the top-p prefix in
    decreasing order, and the relative distance of the draw and of the top-p cut from the
    nearest boundary that would change the token (the decision's rounding margin)."""
    logits = np.asarray(logits, dtype=np.float32)
    V = logits.size
    if temperature <= 0:
        m = logits.max()
        tok = int(np.flatnonzero(logits == m)[0])
        return tok, [tok], np.inf
    k = min(int(top_k), V)
    # decreasing value, ties by increasing index (lexsort orders by its last key first)
    order = [int(i) for i in np.lexsort((np.arange(V), -logits.astype(np.float64)))[:k]]
    l = logits[order].astype(np.float64)
    w = np.exp((l - l[0]) / float(temperature))
    cum = np.zeros(k)
    acc = 0.0
    for i in range(k):  # sequential running sums
        acc += w[i]
        cum[i] = acc
    total = cum[-1]
    need = float(top_p) * total
    n = int(np.flatnonzero(cum >= need)[0]) if top_p < 1.0 else k - 1
    mass = cum[n]
    u = uniform(seed, counter)
    target = u * mass
    j = int(np.flatnonzero(cum[: n + 1] > target)[0])
    lo = cum[j - 1] if j > 0 else 0.0
    margin = min(cum[j] - target, target - lo) / mass
    if top_p < 1.0:  # the cut: the running sums around p * total
        before = cum[n - 1] if n > 0 else 0.0
        margin = min(margin, (cum[n] - need) / total, (need - before) / total if n > 0 else np.inf)
    return order[j], order[: n + 1], margin
