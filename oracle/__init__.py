"""Plain CPU oracle for block-sparse video attention (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline may
import anything here. The CUDA library never calls it and shares no code with
it; its inputs come from ``synth`` (seeded, shared) or from the caller.

Everything is written for a reader to check by eye against the pages:

* ``masks``     - the radial energy-decay mask (Radial Attention news page,
                  hyper.ai) and the LVSA local-window + rotating periodic
                  anchor-frame mask (LVSA review, secrett2633 blog, sec. 3 and
                  Fig. 2), as integer token rules pooled to blocks;
* ``attention`` - textbook masked softmax attention in float64;
* ``kmeans``    - Lloyd k-means used by SVG-EAR's semantic clustering (SVG-EAR,
                  gist.science 2603.08982, technical summary sec. 2, idea 1);
* ``svgear``    - centroid linear compensation, the centroid-proxy error probe
                  and error-to-cost routing under a density budget (same page,
                  sec. 2, ideas 1 and 2).

Parity status: the pages print no worked example or numeric output, so every
function here is pinned by closed forms, invariants, hand-derived cases,
brute force on tiny inputs and independent library routines (tests/), not by
values from the pages.
"""
