"""Write oracle_digests.txt: SHA-256 of the C++ oracle's outputs per workload.

Calls only the CPU oracle (and the seeded input generators).  Run from the
repository root:  python tests/golden/make_digests.py
The digests guard the oracle against silent drift; they are not an input of
any parity test of the CUDA library, which compares against a fresh oracle
run instead.
"""

import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from lidar_point_cloud_gb300 import synth  # noqa: E402

NAMES = ["tiny", "kitti", *[f"uniform_{n}" for n in synth.UNIFORM_SIZES], "dense", "adversarial"]


def digest(name):
    pts, P = synth.make(name)
    st, v, c, n, V = oracle.voxelize(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    assert st == 0
    h = hashlib.sha256()
    for a in (pts, v, c, n):
        h.update(a.tobytes())
    h.update(int(V).to_bytes(4, "little"))
    return V, h.hexdigest()


def main():
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_digests.txt")
    with open(out, "w") as f:
        f.write("# workload V sha256(points || voxels || coords || counts || V)\n")
        f.write("# written by tests/golden/make_digests.py from the CPU oracle\n")
        for name in NAMES:
            V, d = digest(name)
            f.write(f"{name} {V} {d}\n")
            print(name, V, d)


if __name__ == "__main__":
    main()
