"""Per-layer random subset of the visible pages (TEST INFRASTRUCTURE ONLY).

vLLM-Omni RFC "Reconstruction Engine", section 5 ("KV Compression Strategy
Details"): AVGGT samples a random KV subset per layer, different layers drawing
different subsets for coverage; FastVGGT keeps the initial frames' tokens as
global anchors. Read at page granularity on the LingBot-Map visible table
("LingBot-Map Paged KV Cache", section 2): the scale pages (the stream's first
frames) are always kept, and every other visible page is kept with probability
keep / 65536, drawn independently per layer and per position in the table.

The draw for table position e of layer L is the low 16 bits of
splitmix64(seed XOR (L << 32) XOR e); the page is kept when they are below
`keep`. splitmix64 is restated here from its published definition (Steele, Lea
and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014, and
Vigna's reference implementation): this module shares no code with the CUDA
library or with the input generator.
"""

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def splitmix64(state):
    """One splitmix64 output for the 64-bit `state` (the state is advanced by
    the golden gamma, then mixed)."""
    z = (state + GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def page_kept(seed, layer, e, keep):
    """Whether table position e (a non-anchor page) of `layer` is kept."""
    key = (seed ^ (layer << 32) ^ e) & MASK64
    return (splitmix64(key) & 0xFFFF) < keep


def kept_positions(n_entries, n_anchor, seed, layer, keep):
    """Table positions kept, in table order: the first n_anchor always."""
    return [e for e in range(n_entries) if e < n_anchor or page_kept(seed, layer, e, keep)]
