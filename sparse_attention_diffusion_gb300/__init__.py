"""GB300-native MC-Sparse hot path: PDDP query grouping, anchor two-pass exact
top-K selection, token-gather sparse attention and the cached dense-sparse residual.

`mcs` is the thin binding over the C-ABI library `libmcs.so`; `synth` makes the
seeded synthetic layers; `schedule` drives the meta-cache denoising schedule.
"""
