"""Layer shapes that select each tile kernel of the library on a GB300 (152 SMs).

The fused step prefers a CTA pair on 256 x 256 tiles (d_out and d_in multiples of 256), else one
CTA on 128 x 256 (d_in a multiple of 256), else 128 x 128; a layer whose preferred shape would
occupy at most half the SMs (76) takes 128 x 128 tiles instead.  The parity tests name the shape
they exercise and check it through the launch-shape query, so a change of that rule shows there.
"""

PAIR = (2048, 1280)        # 8 x 5 = 40 pair tiles of 256 x 256: 80 CTAs
PAIR_MANY = (4096, 1280)   # 80 pair tiles, more than the 76 pairs resident at once: a persistent tail
WIDE = (1152, 2560)        # d_out not a multiple of 256: 9 x 10 = 90 tiles of 128 x 256
SMALL = (384, 384)         # 9 tiles of 128 x 128
FEW_PAIRS = (512, 768)     # 6 pair tiles would fill 12 SMs: 24 tiles of 128 x 128 instead

TILE = {PAIR: (256, 256, 2), PAIR_MANY: (256, 256, 2), WIDE: (128, 256, 1), SMALL: (128, 128, 1),
        FEW_PAIRS: (128, 128, 1)}
