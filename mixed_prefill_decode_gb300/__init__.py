"""Mixed prefill+decode layer step for GB300 (sm_103a).

The product is the C-ABI library ``libmb.so`` (include/mb.h); ``binding``
marshals arguments to it, ``build`` compiles it in-tree, ``workload`` draws the
seeded synthetic inputs.  Importing the package loads nothing; the library is
loaded on first use of ``binding.lib()`` and fails loudly if it was not built.
"""

__all__ = ["binding", "build", "workload"]
