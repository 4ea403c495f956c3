"""The oracle on all host cores: one process per core, each verifying a
contiguous share of the requests.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the bench's
CPU-baseline leg uses it to time the oracle across the host's cores.  The
oracle itself is unchanged; requests are independent, so a batch splits
into per-process shares with nothing to combine but the outputs.

The inputs sit in POSIX shared memory, written once by the parent.  Each
worker is a separate interpreter (``python -m oracle.pool``) that imports
only numpy and the oracle, attaches to the shared arrays, says ``ready``,
waits for ``go`` on stdin, verifies its share and writes accept_len,
accept_draft and out_token back into shared output arrays.
"""
import json
import os
import subprocess
import sys
import time

import numpy as np

_INPUTS = ("target", "draft", "tokens", "lengths", "accept_u", "sample_u")
_OUTPUTS = ("accept_len", "accept_draft", "out_token")


def _attach(spec):
    from multiprocessing import resource_tracker, shared_memory
    shm = shared_memory.SharedMemory(name=spec["name"])
    # the parent owns the segment: without this, this process's resource
    # tracker would unlink it when the process exits
    resource_tracker.unregister(shm._name, "shared_memory")
    return shm, np.ndarray(tuple(spec["shape"]), dtype=np.dtype(spec["dtype"]), buffer=shm.buf)


def _worker(cfg):
    import oracle
    held = {k: _attach(spec) for k, spec in cfg["arrays"].items()}
    lo, hi = cfg["lo"], cfg["hi"]
    ins = {k: held[k][1][lo:hi] for k in _INPUTS}
    prob = oracle.Problem(ins["target"], ins["draft"], ins["tokens"], ins["lengths"], ins["accept_u"],
                          ins["sample_u"], cfg["temperature"], V=cfg["V"])
    print("ready", flush=True)
    sys.stdin.readline()
    t0 = time.perf_counter()
    out = oracle.verify(cfg["mode"], prob)
    dt = time.perf_counter() - t0
    for k in _OUTPUTS:
        held[k][1][lo:hi] = out[k]
    print(json.dumps({"rc": int(out["rc"]), "seconds": dt}), flush=True)
    shms = [shm for shm, _ in held.values()]
    del prob, ins, out, held  # no view into the segments may outlive them
    for shm in shms:
        shm.close()


def verify_all_cores(arrays, mode, temperature, V, procs=None):
    """Verify a batch (numpy arrays in the library's layout; bf16 logits as
    int16 bits) with one oracle process per core.  Returns (outputs dict,
    wall seconds from the common start to the last worker's end, procs)."""
    from multiprocessing import shared_memory
    B = arrays["target"].shape[0]
    procs = max(1, min(procs or os.cpu_count() or 1, B))
    # shared memory is a tmpfs: writing past its size would kill this
    # process, so check the room first
    need = sum(np.asarray(a).nbytes for a in arrays.values()) + 3 * 4 * B
    st = os.statvfs("/dev/shm")
    if st.f_bavail * st.f_frsize < need + (64 << 20):
        raise RuntimeError(f"/dev/shm has {st.f_bavail * st.f_frsize >> 20} MiB free, {need >> 20} MiB needed")
    shms, specs, workers = [], {}, []
    try:
        for k in _INPUTS + _OUTPUTS:
            a = arrays[k] if k in arrays else np.zeros(B, np.int32)
            a = np.ascontiguousarray(a)
            shm = shared_memory.SharedMemory(create=True, size=max(a.nbytes, 1))
            shms.append(shm)
            np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf)[...] = a
            specs[k] = {"name": shm.name, "shape": list(a.shape), "dtype": a.dtype.str}
        bounds = np.linspace(0, B, procs + 1).astype(int)
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
        for i in range(procs):
            cfg = {"arrays": specs, "lo": int(bounds[i]), "hi": int(bounds[i + 1]), "mode": mode,
                   "temperature": float(temperature), "V": int(V)}
            workers.append(subprocess.Popen([sys.executable, "-m", "oracle.pool", json.dumps(cfg)], cwd=root,
                                            env=env, stdin=subprocess.PIPE, stdout=subprocess.PIPE, text=True))
        for w in workers:
            if w.stdout.readline().strip() != "ready":
                raise RuntimeError("an oracle worker did not start")
        t0 = time.perf_counter()
        for w in workers:
            w.stdin.write("go\n")
            w.stdin.flush()
        results = [json.loads(w.stdout.readline()) for w in workers]
        dt = time.perf_counter() - t0
        for w in workers:
            w.wait()
        if any(r["rc"] != 0 for r in results):
            raise RuntimeError("an oracle worker failed")
        out = {k: np.ndarray(tuple(specs[k]["shape"]), dtype=np.dtype(specs[k]["dtype"]),
                             buffer=shms[len(_INPUTS) + i].buf).copy() for i, k in enumerate(_OUTPUTS)}
        return out, dt, procs
    finally:
        for w in workers:  # none is left waiting on a parent that gave up
            if w.poll() is None:
                w.kill()
                w.wait()
        for shm in shms:
            shm.close()
            shm.unlink()


if __name__ == "__main__":
    _worker(json.loads(sys.argv[1]))
