"""One problem per attention kernel instance, with the instance the planner
must pick for it: (shape (B,T,H,W,NH,HD), kernel, score-tile cap, W stride).

The CPU tests check that each problem selects its instance; the GPU parity
tests run every problem against the oracle, so every compiled instance is
exercised at least once.
"""

INSTANCE_CASES = [
    # default families: 128-key tiles for HD <= 64, 64-key tiles for HD >= 128
    ((1, 5, 13, 23, 2, 64), (3, 5, 9), 128, 14),
    ((1, 5, 13, 23, 2, 64), (3, 5, 7), 128, 12),
    ((1, 4, 8, 16, 2, 64), (1, 1, 1), 128, 16),
    ((1, 4, 16, 5, 2, 64), (1, 1, 1), 128, 8),
    ((1, 4, 8, 24, 2, 64), (1, 1, 7), 128, 32),
    ((1, 4, 8, 33, 2, 64), (1, 1, 11), 128, 0),
    ((1, 4, 8, 33, 2, 64), (1, 1, 33), 128, 1),
    ((1, 6, 16, 14, 2, 128), (3, 3, 5), 64, 12),
    ((1, 6, 16, 20, 2, 128), (3, 3, 5), 64, 14),
    # HD 64, 96-key tiles computed one ahead of the softmax
    ((2, 6, 16, 14, 2, 64), (3, 3, 5), 96, 14),
    ((1, 5, 13, 23, 2, 64), (3, 3, 7), 96, 12),
    ((1, 6, 12, 16, 3, 64), (3, 1, 3), 96, 16),
    ((1, 7, 17, 5, 2, 64), (1, 1, 1), 96, 8),
    ((1, 7, 11, 19, 2, 64), (3, 1, 9), 96, 32),
    ((1, 3, 8, 50, 2, 64), (1, 7, 33), 96, 0),
    # HD 16 and 32, 96-key tiles in pairs of slots
    ((1, 3, 5, 50, 2, 16), (3, 3, 33), 96, 0),
    ((1, 5, 11, 13, 2, 16), (3, 1, 1), 96, 8),
    ((1, 7, 7, 19, 2, 16), (3, 1, 7), 96, 16),
    ((1, 7, 5, 40, 2, 16), (3, 1, 9), 96, 32),
    ((2, 3, 5, 50, 2, 32), (3, 3, 33), 96, 0),
    ((1, 5, 11, 13, 2, 32), (3, 1, 1), 96, 8),
    ((1, 7, 7, 19, 2, 32), (3, 1, 7), 96, 16),
    ((1, 7, 5, 40, 2, 32), (3, 1, 9), 96, 32),
]
