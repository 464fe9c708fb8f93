"""primitive_sm_graph_gb300: the data-parallel hot path of a lazy primitive-op
graph on GB300 (sm_103a).

``_abi`` is the thin ctypes binding of the C ABI in include/psg.h (libpsg.so,
built in-tree by :func:`build.build`).  ``graph`` is the lazy graph builder and
executor that lowers fused groups of primitive nodes onto those calls.
Touching any binding name raises if libpsg.so has not been built: there is no
fallback path.  ``build`` itself imports without the library.
"""
_EXPORTS = ("PsgError", "make_view", "node", "psg_contract", "psg_elementwise", "psg_gather",
            "psg_permute", "psg_query_launch", "psg_reduce_rows", "psg_scatter_add",
            "psg_scatter_workspace", "psg_status_string", "psg_version", "view_of", "RED_MAX",
            "RED_SUM")


def __getattr__(name):
    if name in _EXPORTS:
        from . import _abi
        return getattr(_abi, name)
    raise AttributeError(name)
