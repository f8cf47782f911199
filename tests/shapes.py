"""Layer shapes that select each tile kernel of the library on a GB300 (152 SMs).

The fused step prefers a CTA pair on 256 x 256 tiles (d_out and d_in multiples of 256), else one
CTA on 128 x 256 (d_in a multiple of 256), else 128 x 128; a layer whose preferred shape would
occupy at most half the SMs (76) takes 128 x 128 tiles instead, and if those would too, 128 x 64
tiles (bf16 operands with binary32 or bfloat16 states; INT8 states and E4M3 operands stay on
128 x 128).  With bf16 operands, a pair launch whose last wave would occupy at most half of the 76
pairs runs that wave's tiles as two 256 x 128 halves each (the query still reports 256 x 256).
The parity tests name the shape they exercise and check it through the launch-shape query, so a
change of that rule shows there.
"""

PAIR = (2048, 1280)        # 8 x 5 = 40 pair tiles of 256 x 256: 80 CTAs
PAIR_MANY = (4096, 1280)   # 80 pair tiles for 76 pairs: the last 4 run as 8 half tiles of 256 x 128
WIDE = (1152, 2560)        # d_out not a multiple of 256: 9 x 10 = 90 tiles of 128 x 256
MID = (1536, 1536)         # 36 pair tiles would fill 72 SMs: 144 tiles of 128 x 128
SMALL = (384, 384)         # 9 tiles of 128 x 128 would fill 9 SMs: 18 tiles of 128 x 64
FEW_PAIRS = (512, 768)     # 6 pair tiles, 24 tiles of 128 x 128: 48 tiles of 128 x 64

TILE = {PAIR: (256, 256, 2), PAIR_MANY: (256, 256, 2), WIDE: (128, 256, 1), MID: (128, 128, 1),
        SMALL: (128, 64, 1), FEW_PAIRS: (128, 64, 1)}
