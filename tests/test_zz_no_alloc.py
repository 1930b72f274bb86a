"""ple_lookup_ordered_static: the allocation-free variant of the ordered
gather (fixed per-device scratch inside the library). It must write exactly
what ple_lookup_ordered writes, on two calls in a row (the second reuses the
scratch the first left behind), and refuse sizes beyond its scratch. This
file is collected last so that it also runs after every other test."""

import numpy as np
import pytest
import torch

from hashed_gram_embedding_gb300 import _lib

from _helpers import dev_err_word

pytestmark = pytest.mark.gpu


def _case(seed, rows, T, H, D=128):
    rng = np.random.default_rng(seed)
    table = torch.from_numpy(rng.integers(0, 1 << 16, size=(rows, D), dtype=np.uint16)
                             .view(np.int16)).view(torch.bfloat16)
    ids = rng.integers(0, rows, size=(T, H))
    ids[1, 0] = rows + 3  # outside the table: zero row + flag
    return table, torch.from_numpy(ids).cuda()


@pytest.mark.parametrize("on_host", [False, True])
def test_static_scratch_matches_workspace_version_twice(on_host):
    D = 128
    calls = [_case(1, 70000, 517, 16), _case(2, 9000, 64, 8)]
    owners = []
    for table, ids in calls:
        if on_host:
            owner = _lib.HostTable(table.shape[0], D, torch.bfloat16)
            owner.tensor.copy_(table)
            owners.append(owner)
            tab = owner.tensor
        else:
            tab = table.cuda()
        T, H = ids.shape
        ws = torch.empty((_lib.ple_lookup_ordered_workspace(T, H, tab),), dtype=torch.uint8,
                         device="cuda")
        want = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
        _lib.ple_lookup_ordered(ids, tab, want, ws)
        got = torch.full((T, H * D), 9.0, dtype=torch.bfloat16, device="cuda")
        err = dev_err_word()
        _lib.ple_lookup_ordered_static(ids, tab, got, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) & _lib.PLE_DEVERR_BOUNDS
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    for o in owners:
        o.close()


def test_static_scratch_rejects_oversized_calls():
    rows, D = 1000, 64
    table = torch.zeros((rows, D), dtype=torch.bfloat16, device="cuda")
    T, H = 1 << 20, 4  # 4 Mi items: 16 MiB of walk order > 8 MiB scratch
    ids = torch.zeros((T, H), dtype=torch.int64, device="cuda")
    out = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.PleError, match="static scratch"):
        _lib.ple_lookup_ordered_static(ids, table, out)
