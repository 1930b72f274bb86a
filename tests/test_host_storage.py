"""Host table storage (no GPU): named shared-memory tables (create / attach /
unlink, rollback of every step on failure), file-backed tables mapped
read-only, and the group protocol of open_shared_table over two gloo ranks
-- the leader creates and fills, the other attaches, and any rank's failure
rolls back every rank and unlinks the object. Mappings here are not
registered for the GPU (that needs one; the GPU tests read them over UVA)."""

import os
import socket
import uuid

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from hashed_gram_embedding_gb300 import _lib


@pytest.fixture(scope="module", autouse=True)
def built():
    from hashed_gram_embedding_gb300 import build
    build.build()


def _name():
    return "/ple_test_" + uuid.uuid4().hex[:12]


def _exists(name):
    return os.path.exists("/dev/shm" + name)


def test_create_attach_share_the_rows():
    name = _name()
    a = _lib.MappedHostTable("create", name, 1000, 64, torch.bfloat16, register=False)
    try:
        rows = torch.randn((1000, 64)).to(torch.bfloat16)
        a.tensor.copy_(rows)
        b = _lib.MappedHostTable("attach", name, 1000, 64, torch.bfloat16, register=False)
        assert torch.equal(b.tensor.view(torch.int16), rows.view(torch.int16))
        b.tensor[3, 5] = 7.0  # one object: writes through either mapping
        assert float(a.tensor[3, 5]) == 7.0
        b.close()
    finally:
        a.close()
        _lib.ple_host_table_unlink_shared(name)
    assert not _exists(name)


def test_shared_table_argument_and_state_errors():
    name = _name()
    with pytest.raises(_lib.PleError, match="shm_open"):
        _lib.MappedHostTable("attach", name, 10, 64, torch.bfloat16, register=False)
    for bad in ("no_slash", "/a/b", "/"):
        with pytest.raises(_lib.PleError, match="name"):
            _lib.MappedHostTable("create", bad, 10, 64, torch.bfloat16, register=False)
    a = _lib.MappedHostTable("create", name, 10, 64, torch.bfloat16, register=False)
    try:
        with pytest.raises(_lib.PleError):  # exists already
            _lib.MappedHostTable("create", name, 10, 64, torch.bfloat16, register=False)
        with pytest.raises(_lib.PleError, match="fewer than"):
            _lib.MappedHostTable("attach", name, 11, 64, torch.bfloat16, register=False)
    finally:
        a.close()
        _lib.ple_host_table_unlink_shared(name)
    with pytest.raises(_lib.PleError):
        _lib.ple_host_table_unlink_shared(name)


@pytest.mark.skipif(torch.cuda.is_available(), reason="registration succeeds with a GPU")
def test_failed_registration_rolls_back_the_object():
    # Without a GPU cudaHostRegister fails: the call must undo the mapping and
    # remove the object it created.
    name = _name()
    with pytest.raises(_lib.PleError):
        _lib.MappedHostTable("create", name, 100, 64, torch.bfloat16, register=True)
    assert not _exists(name)


def test_file_backed_table(tmp_path):
    rows = np.random.default_rng(1).integers(0, 1 << 16, size=(500, 64), dtype=np.uint16)
    path = tmp_path / "table.bin"
    rows.tofile(path)
    t = _lib.MappedHostTable("file", path, 500, 64, torch.bfloat16, register=False)
    try:
        assert np.array_equal(t.tensor.view(torch.int16).numpy().view(np.uint16), rows)
    finally:
        t.close()
    with pytest.raises(_lib.PleError, match="fewer than"):
        _lib.MappedHostTable("file", path, 501, 64, torch.bfloat16, register=False)
    with pytest.raises(_lib.PleError, match="open"):
        _lib.MappedHostTable("file", tmp_path / "missing.bin", 1, 64, torch.bfloat16,
                             register=False)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _group_worker(rank, world, port, name, follower_rows, results):
    import torch.distributed as dist
    from hashed_gram_embedding_gb300 import host_storage
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    rows = 256 if rank == 0 else follower_rows
    try:
        t = host_storage.open_shared_table(
            name, rows, 32, torch.float32, group=dist.group.WORLD, register=False,
            fill=lambda x: x.copy_(torch.arange(256 * 32, dtype=torch.float32).view(256, 32)))
        results[rank] = ("ok", float(t.tensor[255, 31]))
        host_storage.close_shared_table(t, name, group=dist.group.WORLD)
    except host_storage.SharedTableError as e:
        results[rank] = ("failed", str(e))
    dist.destroy_process_group()


def _run_group(follower_rows):
    name = _name()
    port = _free_port()
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    procs = [ctx.Process(target=_group_worker, args=(r, 2, port, name, follower_rows, results))
             for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return dict(results), name


def test_group_leader_fills_follower_reads():
    results, name = _run_group(follower_rows=256)
    assert results == {0: ("ok", 256.0 * 32 - 1), 1: ("ok", 256.0 * 32 - 1)}
    assert not _exists(name)


def test_group_rolls_back_when_a_follower_fails():
    # the follower asks for more rows than the object holds: attach fails,
    # every rank raises and the leader removes the object
    results, name = _run_group(follower_rows=257)
    assert results[0][0] == "failed" and results[1][0] == "failed"
    assert "rank 1" in results[0][1] and "fewer than" in results[0][1]
    assert not _exists(name)
