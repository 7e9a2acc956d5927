"""One host copy of the experts for every replica process on a host.

Paged experts need every expert of every layer page-locked in host memory
("Paged Experts", SGLang docs, "Supported Configurations and Limitations").
Replicas that each pinned a private store would need N times that memory; a
48-layer bf16 stack is 58 GB, so a few replicas already exceed a host.  Here
one process creates a shared mapping (a file under /dev/shm, mapped
MAP_SHARED), fills it once, and every replica maps the same pages and hands
them to ``pe_create_external``, which registers them for the device.  The
mapping's pages exist once in host memory whatever the number of replicas.
"""

from __future__ import annotations

import ctypes
import mmap
import os


class SharedHostStore:
    """A MAP_SHARED mapping of ``nbytes`` at ``path`` (created and sized by
    the creator, opened by the others).  ``ptr`` is its address (page
    aligned); keep the object alive while any handle uses it."""

    def __init__(self, path: str, nbytes: int, create: bool):
        flags = os.O_RDWR | (os.O_CREAT | os.O_EXCL if create else 0)
        fd = os.open(path, flags, 0o600)
        try:
            if create:
                os.ftruncate(fd, nbytes)
            elif os.fstat(fd).st_size < nbytes:
                raise ValueError(f"shared store {path} holds {os.fstat(fd).st_size} bytes, need {nbytes}")
            self._mm = mmap.mmap(fd, nbytes, mmap.MAP_SHARED, mmap.PROT_READ | mmap.PROT_WRITE)
        finally:
            os.close(fd)
        self.path, self.nbytes, self.created = path, nbytes, create
        self._anchor = ctypes.c_char.from_buffer(self._mm)
        self.ptr = ctypes.addressof(self._anchor)

    def view(self):
        """The mapping as a writable memoryview (for inspection and tests)."""
        return memoryview(self._mm)

    def close(self, unlink: bool | None = None) -> None:
        """Unmap; the creator also removes the file unless told otherwise."""
        if getattr(self, "_mm", None) is None:
            return
        self._anchor = None
        self._mm.close()
        self._mm = None
        if self.created if unlink is None else unlink:
            try:
                os.unlink(self.path)
            except FileNotFoundError:
                pass


def default_path(tag: str) -> str:
    """A per-run path under /dev/shm (the tag names the job, e.g. its master port)."""
    return os.path.join("/dev/shm", f"pe_store_{tag}")


def open_for_replicas(rep, path: str, nbytes: int, fill) -> SharedHostStore:
    """The replicas' shared store: the replica with local rank 0 creates the
    mapping and calls ``fill(store)`` (loading every expert), then all
    replicas meet at a barrier and the others map the filled store.  Returns
    this replica's mapping; the creator removes the file on ``close()``."""
    from . import replicas

    if rep.local_rank == 0:
        store = SharedHostStore(path, nbytes, create=True)
        try:
            fill(store)
        except BaseException:
            store.close()
            raise
        replicas.barrier(rep)
        return store
    replicas.barrier(rep)
    return SharedHostStore(path, nbytes, create=False)
