"""Plain, slow CPU oracle for the QLoRA NF4 linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import, call or
run anything in this package.  The product path (``bit_quantized_fine_nf4_b300``)
never imports it and shares no code, table or constant generator with it.

Everything here is written from the five QLoRA pages (cited by page title and
section in each docstring), in float64 unless the method fixes float32 (the NF4
encode, the double quantisation of the block scales and the dequantisation are
float32 / bfloat16 by definition, so they are computed in exactly those types).
Where the pages leave a step open the reading taken is stated in the docstring.

Modules
-------
``nf4``     level table, blockwise absmax, NF4 encode / pack, double quantisation,
            dequantisation.
``linear``  LoRA forward / backward through the dequantised weight, SiLU glue.
"""

from . import nf4, linear  # noqa: F401
