"""A PLE table shared by the processes of a group through one /dev/shm object.

PR#56512 report, 关键源码片段: the engram table is kept once per node in a
shared-memory backing file; the group's leader creates it and alone writes
the weights, every process maps it (MAP_SHARED) and registers it with
cudaHostRegister so its GPU reads the rows in place, and a failure anywhere
is broadcast so that every process rolls back. Here the mapping and
registration are libple's (ple_host_table_create_shared / _attach_shared);
this module does the group protocol over a torch.distributed CPU group
(gloo): leader first, its outcome broadcast, then the others, then an
all-gather of every outcome, and a collective rollback (unmap everywhere, the
leader unlinks the object) if any process failed.
"""

import torch.distributed as dist

from . import _lib


class SharedTableError(RuntimeError):
    pass


def open_shared_table(name, rows, row_dim, dtype, group=None, register=True, fill=None):
    """Create (leader, group rank 0) or attach (others) the shared table.

    ``fill(tensor)`` runs on the leader only, before the others attach (the
    leader alone writes the weights). Returns a MappedHostTable on every
    rank, or raises SharedTableError on every rank with each rank's error,
    after undoing all mappings and the object.
    """
    rank = dist.get_rank(group) if group is not None else 0
    table, err = None, None
    if rank == 0:
        try:
            table = _lib.MappedHostTable("create", name, rows, row_dim, dtype, register)
            if fill is not None:
                fill(table.tensor)
        except Exception as e:  # the C call already undid its own steps
            err = f"rank 0: {e}"
            if table is not None:
                table.close()
                _unlink_quietly(name)
                table = None
    if group is not None:
        box = [err]
        dist.broadcast_object_list(box, src=dist.get_global_rank(group, 0), group=group)
        if box[0] is not None:
            raise SharedTableError(box[0])
        if rank != 0:
            try:
                table = _lib.MappedHostTable("attach", name, rows, row_dim, dtype, register)
            except Exception as e:
                err = f"rank {rank}: {e}"
        errors = [None] * dist.get_world_size(group)
        dist.all_gather_object(errors, err, group=group)
        failed = [e for e in errors if e is not None]
        if failed:
            if table is not None:
                table.close()
            dist.barrier(group=group)  # every mapping is gone before the unlink
            if rank == 0:
                _unlink_quietly(name)
            raise SharedTableError("; ".join(failed))
    elif err is not None:
        raise SharedTableError(err)
    return table


def close_shared_table(table, name, group=None):
    """Unmap on every rank; the leader unlinks the object once all are done."""
    table.close()
    rank = dist.get_rank(group) if group is not None else 0
    if group is not None:
        dist.barrier(group=group)
    if rank == 0:
        _unlink_quietly(name)


def _unlink_quietly(name):
    try:
        _lib.ple_host_table_unlink_shared(name)
    except _lib.PleError:
        pass
