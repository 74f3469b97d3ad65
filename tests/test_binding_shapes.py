"""The Python binding's shape checks (no GPU needed): the library receives
bare pointers and sizes, so every tensor shape that the sizes do not imply
must be checked before the call, or a mismatch becomes an out-of-bounds
access on the device."""
import pytest
import torch

from paged_kv_cache_174_gb300 import ops


def _attn(T=5, nq=8, d=64, nb=10, bs=16, nkv=2, S=3, maxb=4):
    return dict(q=torch.empty(T, nq, d), k_cache=torch.empty(nb, bs, nkv, d),
                v_cache=torch.empty(nb, bs, nkv, d), block_tables=torch.empty(S, maxb),
                seq_lens=torch.empty(S), query_start_loc=torch.empty(S + 1))


def test_attention_shapes_accepts_a_consistent_call():
    a = _attn()
    assert ops._attention_shapes(**a) == (5, 8, 64, 10, 16, 2, 3)
    assert ops._attention_shapes(**a, out=torch.empty(5, 8, 64))[0] == 5


@pytest.mark.parametrize("change", [
    dict(q=torch.empty(5, 8, 128)),                    # head_dim differs from the cache
    dict(v_cache=torch.empty(9, 16, 2, 64)),           # v_cache shape differs
    dict(q=torch.empty(5, 7, 64)),                     # n_q not a multiple of n_kv
    dict(query_start_loc=torch.empty(3)),              # not [S + 1]
    dict(block_tables=torch.empty(2, 4)),              # not [S, maxb]
    dict(seq_lens=torch.empty(3, 1)),                  # not 1-D
    dict(q=torch.empty(5, 8)),                         # not [T, n_q, d]
])
def test_attention_shapes_rejects(change):
    a = _attn()
    a.update(change)
    with pytest.raises(ValueError):
        ops._attention_shapes(**a)


def test_attention_shapes_rejects_out_of_another_shape():
    with pytest.raises(ValueError):
        ops._attention_shapes(**_attn(), out=torch.empty(4, 8, 64))


def test_new_rows_shapes():
    k = torch.empty(6, 2, 64)
    ops._new_rows_shapes(k, torch.empty(6, 2, 64), 2, 64, torch.empty(6))
    for v, nkv, d, slots in ((torch.empty(5, 2, 64), 2, 64, torch.empty(6)),   # v rows
                             (torch.empty(6, 2, 64), 4, 64, torch.empty(6)),   # n_kv
                             (torch.empty(6, 2, 64), 2, 128, torch.empty(6)),  # head_dim
                             (torch.empty(6, 2, 64), 2, 64, torch.empty(5))):  # slots
        with pytest.raises(ValueError):
            ops._new_rows_shapes(k, v, nkv, d, slots)


def test_workspace_and_pairs_checks_need_cuda_tensors():
    with pytest.raises(ValueError):
        ops._need_workspace(torch.empty(16, dtype=torch.uint8))   # host memory
    with pytest.raises((TypeError, ValueError)):
        ops._need_pairs(torch.empty(3, 2, dtype=torch.int32))     # host memory
    with pytest.raises(TypeError):
        ops._need_pairs(torch.empty(3, 2, dtype=torch.int64))     # wrong dtype
