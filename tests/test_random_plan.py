"""The seeded random parity sweep (tests/test_gpu_random.py) reaches every
supported shape: checked on the CPU, since drawing the batches needs no GPU."""
from test_gpu_random import N_CASES, _draw


def test_random_draws_cover_every_shape():
    """Every head_dim, group, kv-head count and block size, and both
    decode-only and mixed batches."""
    seen = set()
    kinds = set()
    for seed in range(N_CASES):
        _, decode_only, (d, g, nkv, bs, _, q_lens) = _draw(seed)
        seen |= {("d", d), ("g", g), ("nkv", nkv), ("bs", bs)}
        kinds.add("decode_only" if decode_only else
                  ("mixed" if any(q > 1 for q in q_lens) else "decode"))
    want = {("d", 64), ("d", 128), ("bs", 16), ("bs", 32)}
    want |= {("g", x) for x in (1, 2, 4, 8)} | {("nkv", x) for x in (1, 2, 4, 8)}
    assert want <= seen, want - seen
    assert {"decode_only", "mixed"} <= kinds
